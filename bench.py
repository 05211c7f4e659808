"""Benchmark of one decode step on GB300: append_paged_kv (one new token per
sequence) + batch_decode_paged_kv (gather, RoPE, GQA attention, on-device split
merge), on the Llama-3-8B-shaped bf16 serving load by default.

Prints ONE JSON line (rank 0).  Timing: W warm-up steps, then K timed steps, each
bracketed by CUDA events on the launching stream.  Inputs larger than L2: two replicas
of the workload (same seed, separate device memory) alternate step by step, so a
step's KV is never in L2 (the other replica streamed through it in between), and the
K steps run back to back between one pair of events (value = elapsed / K): the decode
follows the append directly and starts under it (programmatic dependent launch with
PD_DECODE_EARLY_INPUTS), and the next step's append under the decode's tail.  Inputs
that fit in L2: the L2 is flushed before every timed step (a 2x-L2 buffer written,
then another read, leaving it cold and clean) and each step has its own events.  A
second pass of the same steps puts events between the kernels, which times each
kernel alone (decode_us, append_us and the roofline).  The flushed decode time of the
large workloads is reported as well (decode_us_l2_flushed), and so is their decode
launched K times back to back between one pair of events (decode_us_back_to_back: each
launch's start-up under the tail of the one before).  `e2e` re-times the step
through the public API from pinned host buffers (H2D of the step's inputs and D2H of out + lse inside the timed region).
Before each timed pass a spin kernel keeps the device busy while the host enqueues the
pass, so device-side times carry no host launch gaps.

A workload with an external split count (the long-context one) also reports
`multi_stage`: the same decode as page-aligned chunks decoded into fp32 partial states,
then a tree of merge_state_inplace calls, each stage timed with its own events.  The
`cpu_baseline` holds the fp64 oracle timed on one thread and, as `all_cores`, on one
thread per host core.

--impl reference times the fp64 oracle (the CPU baseline) on a bounded sample.
Under torchrun every rank runs its own replica of the workload (no collective on the
data path; weak scaling); the reported time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from paged_kv_decode_19_gb300 import workloads as W  # noqa: E402

# the five serving loads; one bench run times each of them (the headline is --config)
PER_CONFIG = ("tiny_fp32", "llama3_8b_bf16", "long_ctx_bf16", "window_sink_f16",
              "fp8_kv_highconc")
METRIC = "paged decode attention µs/call and KV-read GB/s as % of GB300 HBM peak"
UNIT = "us/call"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# Sources the tensor-core decode's launches depend on (its kernel, the shared device code
# and the host planner); the SIMT kernel, merge/append kernels and the workspace arenas
# do not change what it reads or writes.
_TRAFFIC_EXCLUDE = ("decode_simt.cu", "merge_append.cu", "decode_noalloc.cu", "arena.h")


def _sources_digest() -> str:
    """sha256 over the sources of the tensor-core decode kernel and its host planner
    (identifies the build whose DRAM traffic was measured)."""
    import hashlib
    d = os.path.join(ROOT, "paged_kv_decode_19_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(d)):
        if name.endswith((".cu", ".cuh", ".h")) and name not in _TRAFFIC_EXCLUDE:
            h.update(name.encode())
            h.update(open(os.path.join(d, name), "rb").read())
    return h.hexdigest()


def _measured_traffic(config: str, batch: int):
    """DRAM bytes (read + write) of one decode launch from the committed ncu record, if
    it was taken on the current sources and the same workload; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(f"{config}:B={batch}")
    if not rec or rec.get("sources_sha256") != _sources_digest():
        return None
    return int(rec["dram_bytes_per_launch"])


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _oracle_inputs(wl: W.Workload):
    """The workload's inputs as host arrays, and a function that decodes sequence b
    (all heads) with the oracle.  The oracle is plain C called through ctypes, which
    releases the GIL, so several threads may decode different sequences at once."""
    import oracle
    s = wl.spec
    Q = W.bits(wl.Q)
    pages = W.bits(wl.pages)
    ip = wl.indptr.cpu().numpy()
    vals = wl.values.cpu().numpy()
    li = wl.length_info.cpu().numpy()
    kro = wl.k_rope_pos_offset.cpu().numpy()
    qrp = wl.q_rope_position.cpu().numpy()

    def one(b: int) -> int:
        if s.q_len > 1:
            mask = np.zeros((s.B, s.q_len, s.H_qo), bool)
            mask[b] = True
            oracle.batch_decode_paged_kv_mq(
                Q, pages, ip, vals, li, kro, qrp, q_len=s.q_len, q_dtype=s.q_dtype,
                kv_dtype=s.kv_dtype, H_kv=s.H_kv, page_size=s.page_size,
                rotary_mode=s.rotary_mode, rope_scale=s.rope_scale, rope_theta=s.rope_theta,
                sm_scale=wl.sm_scale, k_scale=wl.k_scale, v_scale=wl.v_scale, mask=mask,
                k_rotated=s.k_rotated)
        else:
            mask = np.zeros((s.B, s.H_qo), bool)
            mask[b] = True
            oracle.batch_decode_paged_kv(
                Q, pages, ip, vals, li, kro, qrp, q_dtype=s.q_dtype, kv_dtype=s.kv_dtype,
                H_kv=s.H_kv, page_size=s.page_size, rotary_mode=s.rotary_mode,
                rope_scale=s.rope_scale, rope_theta=s.rope_theta, sm_scale=wl.sm_scale,
                sliding_window=s.window is not None, k_scale=wl.k_scale, v_scale=wl.v_scale,
                mask=mask, k_rotated=s.k_rotated)
        return int(wl.attended[b])

    return one


def _oracle_sample(wl: W.Workload, budget_s: float):
    """Run the oracle on whole sequences (all heads), one after another, until `budget_s`
    of CPU time is spent; returns (seconds, sequences, attended rows)."""
    one = _oracle_inputs(wl)
    t0 = time.perf_counter()
    nseq = rows = 0
    for b in range(wl.spec.B):
        rows += one(b)
        nseq += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return time.perf_counter() - t0, nseq, rows


def _host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_sample_threads(wl: W.Workload, budget_s: float, threads: int):
    """The same sample with `threads` threads, each decoding whole sequences: the first
    `threads` sequences always run, more are handed out until `budget_s` has passed, and
    the ones already started run to the end.  Returns (wall seconds, sequences, attended
    rows)."""
    import concurrent.futures as cf
    one = _oracle_inputs(wl)
    t0 = time.perf_counter()
    nseq = rows = 0
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        nxt = 0
        running = set()
        while nxt < wl.spec.B or running:
            while (nxt < wl.spec.B and len(running) < threads
                   and (nxt < threads or time.perf_counter() - t0 < budget_s)):
                running.add(ex.submit(one, nxt))
                nxt += 1
            if not running:
                break
            done, running = cf.wait(running, return_when=cf.FIRST_COMPLETED)
            for f in done:
                rows += f.result()
                nseq += 1
    return time.perf_counter() - t0, nseq, rows


def _cpu_baseline(wl: W.Workload, budget_s: float):
    total_rows = int(wl.attended.sum())
    secs, nseq, rows = _oracle_sample(wl, budget_s)
    us_per_call = secs * 1e6 * total_rows / max(rows, 1)
    line = {"value": round(us_per_call, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"fp64 oracle (single thread) on {nseq} of {wl.spec.B} sequences, all "
                      f"{wl.spec.H_qo} heads ({rows} of {total_rows} attended rows) in "
                      f"{secs:.1f} s, scaled to the full batch by attended rows (the decode; "
                      f"the step's append is not timed)"}
    cores = _host_cores()
    if cores > 1:
        secs, nseq, rows = _oracle_sample_threads(wl, budget_s, cores)
        line["all_cores"] = {
            "value": round(secs * 1e6 * total_rows / max(rows, 1), 1), "unit": UNIT,
            "cores": cores,
            "sample": f"the same oracle, unchanged, on {cores} threads (one sequence each at a "
                      f"time): {nseq} of {wl.spec.B} sequences ({rows} of {total_rows} attended "
                      f"rows) in {secs:.1f} s wall, scaled to the full batch by attended rows"}
    return line


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.result = None
        if self.proc is None:
            return
        time.sleep(0.2)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if sm:
            self.result = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                           "reasons": sorted(reasons), "samples": len(sm)}


def _append_inputs(wl: W.Workload, device):
    """New-token K/V for the step's append: q_len tokens per sequence, at rows
    len-q_len .. len-1 (one token, at row len-1, for the single-token decode)."""
    s = wl.spec
    if wl.k_new is not None:
        return wl.k_new, wl.v_new, wl.slot_mapping
    g = torch.Generator(device=device)
    g.manual_seed(12345)
    dt = W.TORCH_DTYPES[s.q_dtype]
    T = s.B * s.q_len
    k = torch.randn((T, s.H_kv, s.D), generator=g, device=device).to(dt)
    v = torch.randn((T, s.H_kv, s.D), generator=g, device=device).to(dt)
    ip = wl.indptr.cpu().numpy()
    vals = wl.values.cpu().numpy()
    row = (wl.seq_len[:, None] - s.q_len + np.arange(s.q_len)[None, :]).reshape(-1)
    seq = np.repeat(np.arange(s.B), s.q_len)
    ok = row >= 0
    rr = np.maximum(row, 0)
    slots = np.where(ok, vals[np.minimum(ip[seq] + rr // s.page_size, max(len(vals) - 1, 0))]
                     .astype(np.int64) * s.page_size + rr % s.page_size, -1)
    return k, v, torch.from_numpy(slots.astype(np.int64)).to(device)


def _external_split(w: "W.Workload", nsplit: int, dev):
    """Inputs of the multi-stage form of a long-context decode: each sequence's page list
    cut into nsplit page-aligned chunks, decoded as nsplit * B pseudo-sequences (chunk
    j of sequence b at j * B + b, Q repeated) into fp32 partial states."""
    s = w.spec
    ipc, valc, lastc, roff = W.split_chunks_padded(w.indptr.cpu().numpy(),
                                                   w.values.cpu().numpy(), w.seq_len,
                                                   s.page_size, nsplit)
    kro = np.tile(w.k_rope_pos_offset.cpu().numpy(), nsplit) + roff
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    n = nsplit * s.B
    return {"Q": w.Q.repeat(nsplit, 1, 1).contiguous(), "indptr": t(ipc), "values": t(valc),
            "length_info": t(lastc), "k_rope_pos_offset": t(kro),
            "q_rope_position": w.q_rope_position.repeat(nsplit).contiguous(),
            "out": torch.empty((n, s.H_qo, s.D), dtype=torch.float32, device=dev),
            "lse": torch.empty((n, s.H_qo), dtype=torch.float32, device=dev)}


def _merge_tree(out, lse, nsplit: int, B: int, merge):
    """log2(nsplit) rounds of the pairwise merge: the first half of the chunk-major
    partial states absorbs the second half, so sequence b ends in row b."""
    half = nsplit
    while half > 1:
        half //= 2
        n = half * B
        merge(out[:n], lse[:n], out[n:2 * n], lse[n:2 * n])
    return out[:B], lse[:B]


def run_external_split(pd, w, x, nsplit: int):
    """The multi-stage decode of one workload: chunk decode, then the merge tree."""
    s = w.spec
    pd.batch_decode_paged_kv(x["Q"], w.pages, x["indptr"], x["values"], x["length_info"],
                             x["k_rope_pos_offset"], x["q_rope_position"], x["out"], x["lse"],
                             s.rotary_mode, s.rope_scale, s.rope_theta, w.sm_scale,
                             k_scale=w.k_scale, v_scale=w.v_scale, num_splits=1)
    return _merge_tree(x["out"], x["lse"], nsplit, s.B, pd.merge_state_inplace)


def run_ours(args, ws, rank, local, config=None):
    import paged_kv_decode_19_gb300 as pd

    config = config or args.config
    over = args.over if config == args.config else {}
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    # Two replicas of the workload (same seed, separate device memory) alternate step by
    # step: when one replica's attended KV exceeds L2, a step never finds its KV in L2
    # (the other replica streamed through L2 in between), without a flush kernel.
    # Smaller workloads flush L2 before every step instead (2x L2 written, then 2x L2
    # read: cold and clean).
    reps = []
    for _ in range(2):
        wl = W.make(config, seed=1000 + rank, device=dev, **over)
        reps.append((wl,) + _append_inputs(wl, dev))
    wl = reps[0][0]
    s = wl.spec
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    alternate = wl.kv_bytes_attended() > l2
    qdims = (s.B,) if s.q_len == 1 else (s.B, s.q_len)
    out = torch.empty(qdims + (s.H_qo, s.D), dtype=W.TORCH_DTYPES[s.out_dtype], device=dev)
    lse = torch.empty(qdims + (s.H_qo,), dtype=torch.float32, device=dev)
    # q_len query tokens per sequence: the multi-query entry point
    decode_api = pd.batch_decode_paged_kv if s.q_len == 1 else pd.batch_decode_paged_kv_mq
    split = dict(num_splits=1) if config == "tiny_fp32" else {}
    stream = torch.cuda.current_stream(dev)
    wbuf = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    rbuf = torch.ones(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)

    def flush_l2():
        # evict the workload from L2 by writing a buffer larger than L2, then read another
        # one so the written lines are written back here rather than inside the timed step
        wbuf.zero_()
        rbuf.amax()

    # a cache that holds K rotated: the append rotates the new rows at their positions
    # (attended index, as the decode's RoPE), the decode then rotates only Q
    kpos = [torch.from_numpy((r[0].k_rope_pos_offset.cpu().numpy()[:, None]
                              + np.maximum(r[0].attended - s.q_len, 0)[:, None]
                              + np.arange(s.q_len)[None, :]).reshape(-1).astype(np.int32)).to(dev)
            for r in reps]
    kpos_of = {id(r[0]): k for r, k in zip(reps, kpos)}

    def append(r):
        w, k_new, v_new, slots = r
        if s.k_rotated:
            pd.append_paged_kv_rope(w.pages, k_new, v_new, slots, kpos_of[id(w)],
                                    s.rotary_mode, s.rope_scale, s.rope_theta, w.k_scale,
                                    w.v_scale)
        else:
            pd.append_paged_kv(w.pages, k_new, v_new, slots, w.k_scale, w.v_scale)

    # host copies of each replica's page-table offsets and lengths (the serving
    # scheduler's own arrays): the decode plans its split from them on the host
    metas = {id(r[0]): pd._lib.host_meta_of(r[0].indptr, r[0].length_info) for r in reps}
    use_host_plan = [True]

    def decode(r):
        # the decode follows the append on the stream: its start-up (page table, Q) may
        # run under the append (PD_DECODE_EARLY_INPUTS)
        w = r[0]
        decode_api(w.Q, w.pages, w.indptr, w.values, w.length_info, w.k_rope_pos_offset,
                   w.q_rope_position, out, lse, s.rotary_mode, s.rope_scale, s.rope_theta,
                   w.sm_scale, k_scale=w.k_scale, v_scale=w.v_scale, early_inputs=True,
                   k_rotated=s.k_rotated, host_meta=metas[id(w)] if use_host_plan[0] else None,
                   **split)

    def prefill(n):
        # a spin kernel of about 60 us per step keeps the device busy (at load clocks)
        # while the host enqueues the n timed steps, so the events time the device work
        # alone, without host launch gaps (outside the timed region)
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(int(max(n, 1) * 60e-6 * 2.0e9))

    def timed_steps(n, flush, breakdown):
        # breakdown=True records an event between append and decode, which times each
        # kernel alone (the decode then no longer starts under the append)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        prefill(n)
        for i in range(n):
            r = reps[i % 2]
            if flush:
                flush_l2()
            e0, e1, e2 = ev[i]
            e0.record(stream)
            append(r)
            if breakdown:
                e1.record(stream)
            decode(r)
            e2.record(stream)
        torch.cuda.synchronize()
        if not breakdown:
            return [e[0].elapsed_time(e[2]) for e in ev], None, None
        return ([e[0].elapsed_time(e[2]) for e in ev], [e[1].elapsed_time(e[2]) for e in ev],
                [e[0].elapsed_time(e[1]) for e in ev])

    for i in range(max(args.warmup, 2)):
        r = reps[i % 2]
        append(r)
        decode(r)
    torch.cuda.synchronize()
    assert pd.check_device_errors() == "PD_OK"
    variant = pd.last_decode_variant()

    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    def timed_run(n):
        # n steps back to back, one event pair around them all: a step's decode may
        # overlap the next step's append and start-up, as in a serving loop
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        prefill(n)
        a.record(stream)
        for i in range(n):
            r = reps[i % 2]
            append(r)
            decode(r)
        b.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) / n]

    with ClockSampler(local) as clk:
        if alternate:
            step_ms = timed_run(args.steps)
        else:  # the flush must stay outside the timed region: one event pair per step
            step_ms, _, _ = timed_steps(args.steps, flush=True, breakdown=False)
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        # the same steps again, each kernel timed alone (decode_us, append_us, roofline)
        _, dec_ms, app_ms = timed_steps(args.steps, flush=not alternate, breakdown=True)
    if ws > 1:
        torch.distributed.barrier()
    assert pd.check_device_errors() == "PD_OK"
    launches = 2 * args.steps
    # the same steps after a flush of L2 (for comparison; not the reported value)
    _, dec_flushed_ms, _ = timed_steps(max(args.steps // 2, 3), flush=True, breakdown=True)
    # the decode planning its split on the device instead (a scan of the device
    # indptr / length_info at the kernel's start), for comparison
    use_host_plan[0] = False
    _, dec_devplan_ms, _ = timed_steps(args.steps, flush=not alternate, breakdown=True)
    use_host_plan[0] = True
    # the decode alone, K launches back to back between one event pair (replicas
    # alternating; only where the inputs exceed L2): each launch's start-up (work split,
    # page table, Q) runs under the tail of the one before, as between the kernels of a
    # serving loop.  Reported beside the per-launch time, which stays the roofline's.
    dec_b2b_ms = None
    if alternate:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        prefill(args.steps)
        a.record(stream)
        for i in range(args.steps):
            decode(reps[i % 2])
        b.record(stream)
        torch.cuda.synchronize()
        dec_b2b_ms = a.elapsed_time(b) / args.steps

    # the multi-stage form of the same decode (for comparison; not the reported value):
    # page-aligned chunks decoded as pseudo-sequences into fp32 partials, then the
    # pairwise merge tree; one event pair around each stage, replicas alternating
    ext = None
    nsplit = s.max_splits
    if nsplit > 1 and s.window is None and s.q_len == 1 and not s.k_rotated:
        assert nsplit & (nsplit - 1) == 0, "the merge tree halves the chunk count"
        xs = [_external_split(r[0], nsplit, dev) for r in reps]
        for i in range(2):
            run_external_split(pd, reps[i][0], xs[i], nsplit)
        n = max(args.steps // 2, 3)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        prefill(n)
        for i in range(n):
            w, x = reps[i % 2][0], xs[i % 2]
            if not alternate:
                flush_l2()
            ev[i][0].record(stream)
            pd.batch_decode_paged_kv(x["Q"], w.pages, x["indptr"], x["values"],
                                     x["length_info"], x["k_rope_pos_offset"],
                                     x["q_rope_position"], x["out"], x["lse"], s.rotary_mode,
                                     s.rope_scale, s.rope_theta, w.sm_scale, k_scale=w.k_scale,
                                     v_scale=w.v_scale, num_splits=1)
            ev[i][1].record(stream)
            _merge_tree(x["out"], x["lse"], nsplit, s.B, pd.merge_state_inplace)
            ev[i][2].record(stream)
        torch.cuda.synchronize()
        assert pd.check_device_errors() == "PD_OK"
        ext = {"nsplit": nsplit,
               "decode_us": statistics.mean(e[0].elapsed_time(e[1]) for e in ev) * 1e3,
               "merge_tree_us": statistics.mean(e[1].elapsed_time(e[2]) for e in ev) * 1e3}
        del xs

    # end-to-end through the public API from pinned host memory: every step copies its
    # inputs (one pinned staging buffer holding Q, the page table, length_info, the RoPE
    # positions and the new tokens' K/V and slots) to the device, runs append + decode on
    # views of that buffer, and reads out + lse back (one buffer); synchronous per step
    names = ("Q", "indptr", "values", "length_info", "k_rope_pos_offset", "q_rope_position")
    srcs = {k: getattr(wl, k) for k in names}
    srcs["k_new"], srcs["v_new"], srcs["slots"] = reps[0][1], reps[0][2], reps[0][3]
    if s.k_rotated:
        srcs["kpos"] = kpos[0]
    offs, total = {}, 0
    for k, t in srcs.items():
        total = (total + 255) // 256 * 256
        offs[k] = total
        total += t.numel() * t.element_size()
    host_in = torch.empty(total, dtype=torch.uint8).pin_memory()
    for k, t in srcs.items():
        nb = t.numel() * t.element_size()
        host_in[offs[k]:offs[k] + nb].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
    dev_in = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]

    def views(buf):
        return {k: buf[offs[k]:offs[k] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                for k, t in srcs.items()}
    dv = [views(b) for b in dev_in]
    out_bytes = out.numel() * out.element_size()
    lse_off = (out_bytes + 255) // 256 * 256
    res_dev = torch.empty(lse_off + lse.numel() * 4, dtype=torch.uint8, device=dev)
    out_e = res_dev[:out_bytes].view(out.dtype).view(out.shape)
    lse_e = res_dev[lse_off:].view(torch.float32).view(lse.shape)
    res_host = torch.empty(res_dev.numel(), dtype=torch.uint8).pin_memory()
    h2d = total
    d2h = res_dev.numel()
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        w, di, buf = reps[i % 2][0], dv[i % 2], dev_in[i % 2]
        if not alternate:
            flush_l2()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        buf.copy_(host_in, non_blocking=True)
        if s.k_rotated:
            pd.append_paged_kv_rope(w.pages, di["k_new"], di["v_new"], di["slots"], di["kpos"],
                                    s.rotary_mode, s.rope_scale, s.rope_theta, w.k_scale,
                                    w.v_scale)
        else:
            pd.append_paged_kv(w.pages, di["k_new"], di["v_new"], di["slots"], w.k_scale,
                               w.v_scale)
        decode_api(di["Q"], w.pages, di["indptr"], di["values"], di["length_info"],
                   di["k_rope_pos_offset"], di["q_rope_position"], out_e, lse_e, s.rotary_mode,
                   s.rope_scale, s.rope_theta, w.sm_scale, k_scale=w.k_scale, v_scale=w.v_scale,
                   early_inputs=True, k_rotated=s.k_rotated, host_meta=metas[id(reps[0][0])],
                   **split)
        res_host.copy_(res_dev, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= args.warmup:
            e2e_ms.append(a.elapsed_time(b))

    # The same step replayed from a CUDA graph, as a serving loop runs it: captured once
    # per replica (the H2D copy, append, decode and D2H copy), the split planned on the
    # device so that the graph reads whatever page table the copy brought; each timed step
    # is one graph launch, the copies still inside the timed region.
    def e2e_step_body(j):
        w, di, buf = reps[j][0], dv[j], dev_in[j]
        buf.copy_(host_in, non_blocking=True)
        if s.k_rotated:
            pd.append_paged_kv_rope(w.pages, di["k_new"], di["v_new"], di["slots"], di["kpos"],
                                    s.rotary_mode, s.rope_scale, s.rope_theta, w.k_scale,
                                    w.v_scale)
        else:
            pd.append_paged_kv(w.pages, di["k_new"], di["v_new"], di["slots"], w.k_scale,
                               w.v_scale)
        decode_api(di["Q"], w.pages, di["indptr"], di["values"], di["length_info"],
                   di["k_rope_pos_offset"], di["q_rope_position"], out_e, lse_e, s.rotary_mode,
                   s.rope_scale, s.rope_theta, w.sm_scale, k_scale=w.k_scale, v_scale=w.v_scale,
                   early_inputs=True, k_rotated=s.k_rotated, **split)
        res_host.copy_(res_dev, non_blocking=True)

    e2e_graph_ms, graph_error = [], None
    try:
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            for j in range(2):  # warm-up on the capture stream (its workspace arena)
                e2e_step_body(j)
        cap.synchronize()
        graphs = []
        for j in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                e2e_step_body(j)
            graphs.append(g)
        torch.cuda.synchronize()
        for i in range(args.warmup + args.steps):
            if not alternate:
                flush_l2()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graphs[i % 2].replay()
            b.record(stream)
            b.synchronize()
            if i >= args.warmup:
                e2e_graph_ms.append(a.elapsed_time(b))
        del graphs
    except Exception as ex:  # a capture the runtime refuses: reported in the line (graph_error)
        graph_error = f"{type(ex).__name__}: {ex}"[:200]
        e2e_graph_ms = []
        torch.cuda.synchronize()
    assert pd.check_device_errors() == "PD_OK"

    res = dict(step=statistics.mean(step_ms), dec=statistics.mean(dec_ms),
               dec_med=statistics.median(dec_ms), app=statistics.mean(app_ms),
               dec_flushed=statistics.mean(dec_flushed_ms),
               dec_devplan=statistics.mean(dec_devplan_ms), dec_b2b=dec_b2b_ms,
               e2e=statistics.mean(e2e_ms),
               e2e_graph=statistics.mean(e2e_graph_ms) if e2e_graph_ms else None,
               graph_error=graph_error,
               launches=launches, variant=variant,
               clocks=clk.result, wl=wl, h2d=h2d, d2h=d2h, alternate=alternate, l2=l2,
               ext=ext)
    return res


def run_cp(args, local, world: int) -> dict:
    """The context-parallel step of the headline load on this GPU, rank by rank: each of
    the `world` ranks' page-aligned slices (pd_cp_shard_plan) decoded into its row of the
    buffer an all-gather would fill (each decode bracketed by its own events), then the
    R-way merge of the gathered partials (pd_merge_states).  Two replicas alternate as in
    the main pass.  The all-gather itself needs `world` GPUs and is not timed."""
    import paged_kv_decode_19_gb300 as pd
    from paged_kv_decode_19_gb300 import cp

    dev = torch.device("cuda", local)
    reps = [W.make(args.config, seed=1000, device=dev, **args.over) for _ in range(2)]
    s = reps[0].spec
    if s.q_len != 1:
        raise ValueError("--cp-ranks: single-token loads only")
    shards = [[cp.shard(w.indptr, w.values, w.length_info, w.k_rope_pos_offset, s.page_size,
                        world, r, dev) for r in range(world)] for w in reps]
    gathered = [torch.empty((world, cp.packed_width(s.B, s.H_qo, s.D)), dtype=torch.float32,
                            device=dev) for _ in reps]
    out = torch.empty((s.B, s.H_qo, s.D), dtype=W.TORCH_DTYPES[s.out_dtype], device=dev)
    lse = torch.empty((s.B, s.H_qo), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def one_step(i, ev=None):
        w, sh, g = reps[i % 2], shards[i % 2], gathered[i % 2]
        for r in range(world):
            if ev is not None:
                ev[r][0].record(stream)
            cp.decode_partial(w.Q, w.pages, sh[r], w.q_rope_position, g[r], s.rotary_mode,
                              s.rope_scale, s.rope_theta, w.sm_scale, k_scale=w.k_scale,
                              v_scale=w.v_scale)
            if ev is not None:
                ev[r][1].record(stream)
        if ev is not None:
            ev[world][0].record(stream)
        cp.combine(g, out, lse)
        if ev is not None:
            ev[world][1].record(stream)

    for i in range(args.warmup):
        one_step(i)
    torch.cuda.synchronize()
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(world + 1)]
           for _ in range(args.steps)]
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(int(args.steps * world * 100e-6 * 2.0e9))
    for i in range(args.steps):
        one_step(i, evs[i])
    torch.cuda.synchronize()
    assert pd.check_device_errors() == "PD_OK"
    rank_us = [statistics.mean(e[r][0].elapsed_time(e[r][1]) for e in evs) * 1e3
               for r in range(world)]
    merge_us = statistics.mean(e[world][0].elapsed_time(e[world][1]) for e in evs) * 1e3
    return {"world": world, "rank_decode_us": [round(x, 2) for x in rank_us],
            "slowest_rank_decode_us": round(max(rank_us), 2), "merge_us": round(merge_us, 2),
            "exchange_bytes_per_rank": cp.packed_width(s.B, s.H_qo, s.D) * 4,
            "what": ("each rank's slice decoded on this GPU in turn (one launch each, events "
                     "around it), then pd_merge_states over the gathered partials; the "
                     "all-gather between GPUs is not timed")}


def _max_or_none(ms, ws: int):
    """Max over ranks of a time in ms (as µs), None where no rank has one.  Every rank
    takes part in the reduction whether or not it has a value, so that a rank without
    one (a graph capture its runtime refused) cannot leave the others waiting."""
    v = _max_over_ranks(ms * 1e3 if ms is not None else -1.0, ws)
    return None if v < 0 else round(v, 2)


def _max_over_ranks(x: float, ws: int) -> float:
    """Max of x over the ranks of the default process group (the replicas' times)."""
    if ws == 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="llama3_8b_bf16", choices=list(W.SPECS))
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle time for the CPU baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time the --config workload alone (no per_config block)")
    ap.add_argument("--B", type=int, default=None,
                    help="override the batch size (smaller cases for profiling)")
    ap.add_argument("--page-size", type=int, default=None,
                    help="override the page size (the pool keeps its row count)")
    ap.add_argument("--q-len", type=int, default=None,
                    help="override the query tokens per sequence (multi-query decode)")
    ap.add_argument("--cp-ranks", type=int, default=0,
                    help="also time the context-parallel step of the headline load for this "
                         "many ranks, rank by rank on this GPU (field context_parallel)")
    args = ap.parse_args()
    args.over = {} if args.B is None else {"B": args.B}
    if args.q_len is not None:
        args.over["q_len"] = args.q_len
    if args.page_size is not None:
        base = W.spec(args.config)
        args.over["page_size"] = args.page_size
        if isinstance(base.pool, int):
            args.over["pool"] = base.pool * base.page_size // args.page_size
    args.warmup = max(args.warmup, 3)
    ws, rank, local = _dist()
    spec = W.spec(args.config, **args.over)
    cfg = {"workload": f"{args.config}: B={spec.B}, H_qo={spec.H_qo}, H_kv={spec.H_kv}, "
                       f"D={spec.D}, page_size={spec.page_size}, {spec.kv_dtype} KV",
           "B": spec.B, "H_qo": spec.H_qo, "H_kv": spec.H_kv, "D": spec.D,
           "page_size": spec.page_size, "kv_dtype": spec.kv_dtype, "q_dtype": spec.q_dtype,
           "rotary_mode": spec.rotary_mode, "len_dist": list(spec.len_dist), "q_len": spec.q_len,
           "step": ("append_paged_kv_rope (1 token/seq, K rotated) + batch_decode_paged_kv "
                    "(PD_DECODE_K_ROTATED)" if spec.k_rotated else
                    "append_paged_kv (1 token/seq) + batch_decode_paged_kv" if spec.q_len == 1 else
                    f"append_paged_kv ({spec.q_len} tokens/seq) + batch_decode_paged_kv_mq "
                    f"(q_len={spec.q_len}, causal among the new tokens)"),
           "l2": None,  # filled in below
           "parallelism": f"replicas x{ws} (each rank its own batch; no collective)"}

    if args.impl == "reference":
        if rank != 0:
            return
        cfg["l2"] = "not applicable (the fp64 oracle on the host cores)"
        wl = W.make(args.config, seed=1000, **args.over)
        for _ in range(args.warmup):
            _oracle_sample(wl, 0.0)
        times, secs_timed, rows_timed = [], 0.0, 0
        for _ in range(args.steps):
            secs, nseq, rows = _oracle_sample(wl, 0.0)  # one sequence per step
            times.append(secs * 1e6 * int(wl.attended.sum()) / max(rows, 1))
            secs_timed += secs
            rows_timed += rows
        v = statistics.mean(times)
        line = {"metric": METRIC, "value": round(v, 1), "unit": UNIT, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(v / 1e3, 3),
                "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic", "config": cfg, "impl": "reference",
                "cpu_baseline": {"value": round(v, 1), "unit": UNIT, "cores": 1,
                                 "kind": "oracle",
                                 "sample": "fp64 oracle, single thread: each step decodes one "
                                           "sequence (all heads) and is scaled to the batch by "
                                           "attended rows; the step's append (one row per "
                                           "sequence) is not timed"},
                "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0},
                # the value is not a measured whole call: each step times one sequence and
                # scales it to the batch by attended rows
                "value_is_scaled": True,
                "scaling_of_value": {"rows_per_call": int(wl.attended.sum()),
                                     "rows_timed_per_step": round(rows_timed / max(args.steps, 1), 1),
                                     "seconds_timed_per_step": round(secs_timed / max(args.steps, 1), 3)}}
        print(json.dumps(line))
        return

    if ws > 1:
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, ws, rank, local)
    head = _summarise(res, args.config, spec, ws)
    # the other serving loads, each in its own pass (their own replicas, warm-up and
    # timed steps), reported beside the headline in `per_config`
    per = {}
    if not args.no_per_config:
        for name in PER_CONFIG:
            if name == args.config:
                continue
            torch.cuda.empty_cache()
            r = run_ours(args, ws, rank, local, config=name)
            per[name] = _summarise(r, name, W.spec(name), ws)
            del r
    if rank != 0:
        torch.distributed.destroy_process_group() if ws > 1 else None
        return
    wl = res["wl"]
    cfg["l2"] = head.pop("l2")
    cfg["timing"] = ("CUDA events on the launching stream; each timed pass is enqueued "
                     "behind a spin kernel, so it runs without host launch gaps")
    line = {
        "metric": METRIC,
        # per-call time of the step (append + decode), the slowest replica's: every rank
        # decodes its own full batch, so the time per call does not shrink with N
        "value": head["step_us"],
        "unit": UNIT,
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(head["step_us"] / 1e3, 5),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": spec.kv_dtype,
        "data": "synthetic",
        "config": cfg,
        "decode_us": head["decode_us"],
        "decode_us_l2_flushed": head["decode_us_l2_flushed"],
        "decode_us_device_plan": head["decode_us_device_plan"],
        "decode_us_back_to_back": head["decode_us_back_to_back"],
        "append_us": head["append_us"],
        "kv_read_gbs": head["kv_read_gbs"],
        "decode_variant": head["decode_variant"],
        "roofline": head["roofline"],
        "e2e": head["e2e"],
        "gpu_launches": res["launches"] + sum(p["gpu_launches"] for p in per.values()),
        "clocks": head["clocks"],
    }
    if ws > 1:
        line["aggregate_calls_per_s"] = round(ws * 1e6 / head["step_us"], 1)
    if "multi_stage" in head:
        line["multi_stage"] = head["multi_stage"]
    if per:
        line["per_config"] = per
    if args.cp_ranks > 1 and ws == 1:
        line["context_parallel"] = run_cp(args, local, args.cp_ranks)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = _cpu_baseline(wl, args.cpu_budget)
    print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()


def _summarise(res, config: str, spec, ws: int) -> dict:
    """The bench numbers of one workload's pass (times are the maximum over ranks)."""
    step_us = _max_over_ranks(res["step"] * 1e3, ws)
    dec_us = _max_over_ranks(res["dec"] * 1e3, ws)
    e2e_us = _max_over_ranks(res["e2e"] * 1e3, ws)
    wl = res["wl"]
    kv_bytes = wl.kv_bytes_attended()
    alg_bytes = kv_bytes + wl.io_bytes()
    peak, peak_kind = _peaks()
    achieved = alg_bytes / (dec_us * 1e-6) / 1e9
    out = {
        "workload": f"{config}: B={spec.B}, H_qo={spec.H_qo}, H_kv={spec.H_kv}, D={spec.D}, "
                    f"page_size={spec.page_size}, {spec.kv_dtype} KV",
        "step_us": round(step_us, 2),
        "decode_us": round(dec_us, 2),
        "decode_us_l2_flushed": round(res["dec_flushed"] * 1e3, 2),
        "decode_us_device_plan": round(_max_over_ranks(res["dec_devplan"] * 1e3, ws), 2),
        "decode_us_back_to_back": (None if res.get("dec_b2b") is None else
                                   round(_max_over_ranks(res["dec_b2b"] * 1e3, ws), 2)),
        "append_us": round(res["app"] * 1e3, 2),
        "kv_read_gbs": round(kv_bytes / (dec_us * 1e-6) / 1e9, 1),
        "decode_variant": res["variant"],
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": _measured_traffic(config, spec.B),
                     "kernel": f"decode_{res['variant']}_kernel",
                     "algorithmic_bytes": alg_bytes, "peak_source": f"{peak_kind} hbm_gbs"},
        "e2e": {"value": round(e2e_us, 2), "unit": UNIT,
                "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                "graph_replayed": _max_or_none(res.get("e2e_graph"), ws)},
        **({"graph_error": res["graph_error"]} if res.get("graph_error") else {}),
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
        "l2": (f"inputs larger than L2 ({kv_bytes / 1e6:.0f} MB attended KV vs "
               f"{res['l2'] / 1e6:.0f} MB L2): two replicas alternate, no flush; the "
               "steps run back to back between one pair of events"
               if res["alternate"] else
               "flushed before every timed step: 2x L2 written, then 2x L2 read (cold, clean L2)"),
    }
    if res["ext"]:
        e = res["ext"]
        out["multi_stage"] = {
            "chunks": e["nsplit"], "decode_us": round(e["decode_us"], 2),
            "merge_tree_us": round(e["merge_tree_us"], 2),
            "total_us": round(e["decode_us"] + e["merge_tree_us"], 2),
            "what": (f"each sequence cut into {e['nsplit']} page-aligned chunks, decoded as "
                     f"{e['nsplit']} x B pseudo-sequences into fp32 partial states (one "
                     f"launch), then {e['nsplit'].bit_length() - 1} rounds of "
                     "merge_state_inplace; compare decode_us (the split merged inside the "
                     "decode launch)")}
    return out


if __name__ == "__main__":
    main()
