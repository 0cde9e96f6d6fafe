#!/usr/bin/env python
"""Benchmark of the sparse-decode KV offload step on GB300.

One step = one pass of the whole hot path over the batch: append the new
tokens (rows to the pinned host pool, keys to the indexer cache), then
kvo_step (score every cached token, fused top-k with packed payload, MTP
merge/dedup, LRU residency update, miss-row fill from host, remap).

Workload (default): the largest single-GPU configuration, 32 requests x 16
layers, 65,536-token context, top-2048 of a 16,384-slot hot shelf (a quarter
of the context), one query position, random-walk queries with drift 0.95, a
50-step decode sequence, 38.7 GB of main KV in the pinned host pool.  The
warm-up steps run the start of the sequence; the timed steps continue it (past
step 49 every unit is returned to its prefilled tokens with an empty shelf,
kvo_reset, and the sequence starts again).  The cold step (an empty shelf, every
selected row a miss) is timed on its own after the timed steps.  The 8.59 GB of
indexer keys read per step exceed the 129 MB L2.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle instead.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode steps/s (layer·request selections/s) + miss-fill GB/s vs roofline"
UNIT = "selections/s"
DEFAULT_WORKLOAD = "batch32x16_64k"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_HBM_GBS = 6800.0


# --------------------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(backend):
    import torch.distributed as dist
    world, rank, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return world, rank


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x, world, device=None):
    """Max of a float over ranks (identity when world == 1)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, steps, max_ms, world):
    """Selections per second of all ranks: every rank processes units_per_rank x steps."""
    return units_per_rank * steps * world / (max_ms / 1e3)


# --------------------------------------------------------------------------- helpers
def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


FALLBACK_BF16_TFLOPS = 1900.0


def load_bf16_peak():
    """Dense bf16 tensor peak (TFLOP/s) for a kernel timed on its own: the burst figure."""
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def huge_backed_fraction(addr):
    """Fraction of the mapping that holds host address addr backed by transparent huge
    pages (from /proc/self/smaps), or None when it cannot be read."""
    try:
        with open("/proc/self/smaps") as f:
            lines = f.read().splitlines()
    except OSError:
        return None
    for i, line in enumerate(lines):
        head = line.split()
        if not head or "-" not in head[0]:
            continue
        try:
            lo, hi = (int(x, 16) for x in head[0].split("-"))
        except ValueError:
            continue
        if lo <= addr < hi:
            size = anon_huge = None
            for l2 in lines[i + 1:i + 40]:
                if l2.startswith("Size:"):
                    size = int(l2.split()[1])
                elif l2.startswith("AnonHugePages:"):
                    anon_huge = int(l2.split()[1])
                if size is not None and anon_huge is not None:
                    return round(anon_huge / size, 4) if size else None
            return None
    return None


def numa_spread(addr):
    """Share of the pages of the mapping that holds host address addr on each NUMA node
    (from /proc/self/numa_maps), e.g. {"N0": 1.0}, or None when it cannot be read.  Where
    a pinned pool sits decides how fast the host link can read it."""
    try:
        with open("/proc/self/numa_maps") as f:
            lines = f.read().splitlines()
    except OSError:
        return None
    best = None
    for line in lines:
        parts = line.split()
        try:
            start = int(parts[0], 16)
        except (ValueError, IndexError):
            continue
        if start <= addr and (best is None or start > best[0]):
            best = (start, parts)
    if best is None:
        return None
    counts = {}
    for tok in best[1]:
        if tok.startswith("N") and "=" in tok and tok[1:tok.index("=")].isdigit():
            counts[tok[:tok.index("=")]] = int(tok[tok.index("=") + 1:])
    total = sum(counts.values())
    return {n: round(c / total, 4) for n, c in sorted(counts.items())} if total else None


def gpu_numa_node(index):
    """NUMA node of GPU `index` from sysfs (via its PCI bus id), or None."""
    try:
        out = subprocess.run(["nvidia-smi", "-i", str(index), "--query-gpu=pci.bus_id",
                              "--format=csv,noheader"], capture_output=True, text=True, timeout=20)
        bus = out.stdout.strip().lower()
        dom, rest = bus.split(":", 1)
        with open("/sys/bus/pci/devices/%s:%s/numa_node" % (dom[-4:], rest)) as f:
            n = int(f.read().strip())
        return n if n >= 0 else None
    except (OSError, ValueError, subprocess.SubprocessError):
        return None


# Kernels bracketed with CUDA events inside the timed region: those a roofline is reported for.
TIMED_KINDS = ("score", "gather", "fused")


def _kinds_mask(names):
    from top_cache_gb300 import kvo as K
    return sum(1 << K.PROF_KINDS.index(n) for n in names)


# The sources each timed kernel is compiled from (its translation unit and every header it
# includes): a committed traffic figure stands only while their hash is the one it was taken at.
KERNEL_SOURCES = {
    "fused": ["kvo_fused.cu", "kvo_fused_i8.cu", "kvo_fused.cuh", "kvo_device.cuh", "kvo_internal.cuh"],
    "score": ["kvo_select.cu", "kvo_device.cuh", "kvo_internal.cuh"],
    "append": ["kvo_residency.cu", "kvo_device.cuh", "kvo_internal.cuh"],
    "gather": ["kvo_residency.cu", "kvo_device.cuh", "kvo_internal.cuh"],
    "attend": ["kvo_attend.cu", "kvo_internal.cuh"],
}


def kernel_sources(kernel):
    """Repository paths of the files kernel is compiled from (the C ABI header included)."""
    return ["top_cache_gb300/csrc/" + f for f in KERNEL_SOURCES[kernel]] + ["include/kvo.h"]


def code_only(text):
    """C/C++ source without its comments, trailing blanks and empty lines: what the compiler
    sees, so that an edit to a comment leaves a traffic figure's hash unchanged."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    for rel in kernel_sources(kernel):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def load_traffic(kernel, workload):
    """Per-launch DRAM bytes of kernel from the committed ncu summary, if it is current."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        e = t[kernel]
        if e.get("source_hash") != kernel_source_hash(kernel) or e.get("workload") != workload:
            return None
        return float(e["bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples (host-timestamped) while the GPU runs the timed steps."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, period_ms=100):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        win = [p for (t, p) in self.samples if t0 <= t <= t1]
        used = "timed region"
        if len(win) < 3:
            win = [p for (_, p) in self.samples]
            used = "timed region and the clock window right after it"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [num(p[1]) for p in win if num(p[1]) is not None]
        mx = [num(p[2]) for p in win if num(p[2]) is not None]
        pw = [num(p[3]) for p in win if num(p[3]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for p in win for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(win), "window": used}


def measure_host_link(torch, device, nbytes=1 << 30, reps=5):
    """Copy-engine bandwidth pinned host <-> device (GB/s), best of reps."""
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device=device)
    h.fill_(1)
    out = {}
    for name, fn in (("h2d", lambda: d.copy_(h, non_blocking=True)),
                     ("d2h", lambda: h.copy_(d, non_blocking=True))):
        best = 0.0
        for _ in range(reps):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            s.record()
            fn()
            e.record()
            torch.cuda.synchronize()
            best = max(best, nbytes / (s.elapsed_time(e) / 1e3) / 1e9)
        out[name] = best
    del h, d
    torch.cuda.empty_cache()
    return out


# --------------------------------------------------------------------------- workload set-up
def make_workload(args):
    import workload as W
    wl = W.WORKLOADS[args.workload]
    kw = {}
    if args.requests:
        kw["n_requests"] = args.requests
    if args.layers:
        kw["n_layers"] = args.layers
    if args.context:
        kw["context"] = args.context
    if args.drift is not None:
        kw["drift"] = args.drift
    if kw:
        wl = W.reduced(wl, **kw)
    return wl


def prepare(wl, rank, device, log, idx="bf16", block_tokens=0):
    """Handle with the prefilled context, plus per-sequence-step inputs on the device."""
    import numpy as np
    import torch
    import workload as W
    from top_cache_gb300 import kvo as K

    units = [(rank * wl.n_requests + r, l) for r in range(wl.n_requests) for l in range(wl.n_layers)]
    U = len(units)
    S = wl.steps
    tmax = wl.max_tokens(S)
    t0 = time.time()
    kv = K.Kvo(wl.n_requests, wl.n_layers, tmax, wl.topk, wl.hot_capacity, wl.n_pos, wl.row_elems,
               device=device.index or 0, idx_dtype=K.KVO_IDX_INT8 if idx == "int8" else K.KVO_IDX_BF16,
               host_block_tokens=block_tokens)
    if block_tokens:
        # paged pool: every unit's blocks scattered through the pool (seeded permutation)
        mb = -(-tmax // block_tokens)
        tables = np.random.default_rng(wl.seed).permutation(U * mb).astype(np.int32).reshape(U, mb)
        for u in range(U):
            kv.set_blocks(u, tables[u])
            for j in range(-(-wl.context // block_tokens)):
                t = j * block_tokens
                W.token_rows_into(kv.host_block(int(tables[u][j])), 0, wl.seed, W.KIND_ROWS, [units[u]], t,
                                  min(block_tokens, wl.context - t), wl.row_elems)
    else:
        unit_stride = (kv.host_rows(1) - kv.host_rows(0)) // 2 if U > 1 else 0
        W.token_rows_into(kv.host_rows(0), unit_stride, wl.seed, W.KIND_ROWS, units, 0, wl.context,
                          wl.row_elems)
    chunk = max(1, (256 << 20) // max(1, wl.context * 256))
    for b in range(0, U, chunk):
        ids = list(range(b, min(U, b + chunk)))
        keys = torch.from_numpy(W.token_rows(wl.seed, W.KIND_KEYS, [units[u] for u in ids], 0,
                                             wl.context, 128)).to(device)
        for j, u in enumerate(ids):
            kv.prefill(u, wl.context, keys[j])
        torch.cuda.synchronize(device)
        del keys
    # inputs of every step of the sequence (untimed set-up)
    rows = np.empty((S, U, wl.n_new, wl.row_elems), np.uint16)
    keys = np.empty((S, U, wl.n_new, 128), np.uint16)
    for s in range(S):
        t = wl.context + s * wl.n_new
        rows[s] = W.token_rows(wl.seed, W.KIND_ROWS, units, t, wl.n_new, wl.row_elems)
        keys[s] = W.token_rows(wl.seed, W.KIND_KEYS, units, t, wl.n_new, 128)
    q = W.unit_queries(wl.seed, units, wl.drift, S, wl.n_pos)
    inp = {"rows_h": rows, "keys_h": keys, "q_h": q,
           "rows": torch.from_numpy(rows).to(device), "keys": torch.from_numpy(keys).to(device),
           "q": torch.from_numpy(q).to(device)}
    log("set-up %.1f s (host pool %.2f GB pinned)" % (time.time() - t0,
                                                        U * tmax * wl.row_elems * 2 / 1e9))
    return kv, inp, units


class Sequence:
    """Replays the workload's decode sequence: reset to the prefill every S steps."""

    def __init__(self, kv, inp, wl):
        self.kv, self.inp, self.wl = kv, inp, wl
        self.g = 0

    def pos(self):
        return self.g % self.wl.steps

    def step(self, out=None):
        p = self.pos()
        if p == 0 and self.g > 0:
            self.kv.reset(self.wl.context)
        self.kv.append(self.inp["rows"][p], self.inp["keys"][p])
        self.kv.step(self.inp["q"][p], out=out)
        self.g += 1
        return p


# --------------------------------------------------------------------------- attention
def run_attention(args, kv, wl, units, device, torch):
    """Time kvo_attend (decode step 7) on the slots of the last step, on its own.

    Algorithmic work per (unit, position): 2 * H * n * (576 + 512) FLOPs for n listed rows
    (scores over the full row, values over the latent part).  The kernel's CTA pair splits
    the scores by slab, so it executes exactly that."""
    import numpy as np
    import workload as W
    H = args.attend_heads
    P, k = wl.n_pos, wl.topk
    U = len(units)
    q = W.attention_queries(wl.seed, units, 0, P, H)
    qd = torch.from_numpy(q.view(np.int16)).to(device)
    del q
    out = torch.empty((U, P, H, 512), dtype=torch.bfloat16, device=device)
    lse = torch.empty((U, P, H), dtype=torch.float32, device=device)
    slots = kv.slots[:U]
    n_rows = int(((slots >= 0) & (slots < wl.hot_capacity)).sum().item())
    scale = 1.0 / (192.0 ** 0.5)
    stream = torch.cuda.current_stream(device)
    for _ in range(3):
        kv.attend(qd, scale, out, lse)
    torch.cuda.synchronize(device)
    n_launch = args.attend_launches
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_launch)]
    for i in range(n_launch):
        ev[2 * i].record(stream)
        kv.attend(qd, scale, out, lse)
        ev[2 * i + 1].record(stream)
    torch.cuda.synchronize(device)
    st = kv.stats()
    ms = [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(n_launch)]
    t = statistics.mean(ms)
    flops = 2.0 * H * n_rows * (576 + 512)
    flops_exec = flops
    peak, src = load_bf16_peak()
    achieved = flops / (t * 1e-3) / 1e12
    # each CTA of a pair reads its own slabs: the pair reads every listed row once
    rows_bytes = U * P * (H // 128) * k * 1152 + U * P * H * 576 * 2
    return {
        "kernel": "attend_kernel", "heads": H, "scale": round(scale, 6), "launches": n_launch,
        "ms_per_launch": round(t, 4), "ms_min": round(min(ms), 4),
        "selections_per_s": round(U / (t * 1e-3), 1),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "peak_source": "%s bf16 dense (burst)" % src,
                     "traffic": load_traffic("attend", wl.name)},
        "flops_per_launch": flops, "executed_tflops": round(flops_exec / (t * 1e-3) / 1e12, 1),
        "rows_listed": n_rows, "l2_to_sm_bytes_per_launch": rows_bytes,
        "l2": "inputs larger than L2: %.2f GB of listed hot rows and queries per launch"
              % (rows_bytes / 1e9),
        "timeouts": st["timeouts"],
    }


def run_copy_sfa(args, kv, inp, wl, units, device, torch):
    """Decode step + sparse attention over the whole sequence, two ways: the step fills the
    miss rows and the attention kernel runs after it ("serial"), or the step leaves them and
    the attention kernel reads them from the pinned pool itself and writes them to their
    slots ("deferred", KVO_OPT_DEFER_FILL; the pages' Copy-SFA operator).  Each way replays
    the sequence from the prefill; the medians of the warm steps are compared.  The
    fraction of the fill hidden is (serial - deferred) / (step with fill - step without)."""
    import numpy as np
    import workload as W
    from top_cache_gb300 import kvo as K
    H = args.attend_heads
    P = wl.n_pos
    U = len(units)
    q = W.attention_queries(wl.seed, units, 0, P, H)
    qd = torch.from_numpy(q.view(np.int16)).to(device)
    del q
    out = torch.empty((U, P, H, 512), dtype=torch.bfloat16, device=device)
    lse = torch.empty((U, P, H), dtype=torch.float32, device=device)
    scale = 1.0 / (192.0 ** 0.5)
    stream = torch.cuda.current_stream(device)
    res = {}
    for name, defer in (("serial", 0), ("deferred", 1)):
        kv.set_option(K.KVO_OPT_DEFER_FILL, defer)
        kv.reset(wl.context)
        seq = Sequence(kv, inp, wl)
        n = wl.steps
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3 * n)]
        st0 = kv.stats()
        for i in range(n):
            ev[3 * i].record(stream)
            seq.step()
            ev[3 * i + 1].record(stream)
            kv.attend(qd, scale, out, lse)
            ev[3 * i + 2].record(stream)
        torch.cuda.synchronize(device)
        st1 = kv.stats()
        step = [ev[3 * i].elapsed_time(ev[3 * i + 1]) for i in range(1, n)]
        att = [ev[3 * i + 1].elapsed_time(ev[3 * i + 2]) for i in range(1, n)]
        tot = [ev[3 * i].elapsed_time(ev[3 * i + 2]) for i in range(1, n)]
        res[name] = {"step_ms": round(statistics.median(step), 4), "attend_ms": round(statistics.median(att), 4),
                     "total_ms": round(statistics.median(tot), 4),
                     "cold_total_ms": round(ev[0].elapsed_time(ev[2]), 4),
                     "rows_h2d_per_step": (st1["rows_h2d"] - st0["rows_h2d"]) / n,
                     "dup_host_bytes_per_step": (st1["fetch_dup_bytes"] - st0["fetch_dup_bytes"]) / n,
                     "timeouts": st1["timeouts"]}
    kv.set_option(K.KVO_OPT_DEFER_FILL, 0)
    kv.reset(wl.context)
    fill = res["serial"]["step_ms"] - res["deferred"]["step_ms"]
    saved = res["serial"]["total_ms"] - res["deferred"]["total_ms"]
    res["fill_ms"] = round(fill, 4)
    res["hidden_fraction"] = round(saved / fill, 4) if fill > 0 else None
    res["selections_per_s"] = {k_: round(U / (res[k_]["total_ms"] * 1e-3), 1) for k_ in ("serial", "deferred")}
    return res


# --------------------------------------------------------------------------- layerwise prefill
def run_layerwise(args, link, device, torch, log):
    """Time prefill passes of the layerwise offload (kvo_lw_*) on their own.

    Per pass and layer: the cached prefix is loaded into the layer's buffer (unless it is
    resident), a stand-in compute of a fixed window runs on the caller's stream (a timed
    spin, so that it takes no memory bandwidth, then the copy of the chunk's rows into the
    buffer), and the chunk's rows are saved to the host pool.  Roofline of a pass: the
    slower of the compute windows and each link direction at its measured peak."""
    import numpy as np
    import workload as W
    from top_cache_gb300 import kvo as K
    N, L0, c, n_pass = args.lw_layers, args.lw_prefix, args.lw_chunk, args.lw_passes
    row = 576
    T = L0 + c * (n_pass + 1)
    t0 = time.time()
    lw = K.Layerwise(N, T, 1, 3, 1, row)
    try:
        for l in range(N):
            W.token_rows_into(lw.host_rows_ptr(l), 0, 3001, W.KIND_ROWS, [(0, l)], 0, L0, row)
        lw.set_length(L0)
        chunk = torch.zeros((c, row), dtype=torch.int16, device=device)
        # compute window per layer: the load time of the mid-run prefix at the measured peak
        # (the pages' condition for a free transfer: window >= copy time)
        L_mid = L0 + c * (n_pass // 2)
        win_us = args.lw_window_us or (L_mid * row * 2 / (link["h2d"] * 1e9) * 1e6)
        stream = torch.cuda.current_stream(device)
        # calibrate the spin: cycles per microsecond at the current clock
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(1000000)
        c0.record(stream)
        torch.cuda._sleep(2000000)
        c1.record(stream)
        torch.cuda.synchronize(device)
        cycles = int(win_us * 2000000 / (c0.elapsed_time(c1) * 1e3))
        scratch = torch.empty_like(chunk)

        def one_pass(L):
            lw.begin(c)
            for l in range(N):
                buf = lw.layer(l)
                torch.cuda._sleep(cycles)
                buf[L:L + c].copy_(chunk)
                lw.layer_done(l)
            lw.end()

        huge_frac = huge_backed_fraction(lw.host_rows_ptr(0))
        pool_numa = numa_spread(lw.host_rows_ptr(0))
        log("layerwise set-up %.1f s (host pool %.2f GB)" % (time.time() - t0, N * T * row * 2 / 1e9))
        # two warm-up passes over the same prefix (the first timed pass after a single one
        # has been seen to take up to ten times the others, once per process)
        for _ in range(2):
            lw.set_length(L0)
            one_pass(L0)
        torch.cuda.synchronize(device)
        st0 = lw.stats()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_pass + 1)]
        ev[0].record(stream)
        L = L0 + c
        for i in range(n_pass):
            one_pass(L)
            L += c
            ev[i + 1].record(stream)
        torch.cuda.synchronize(device)
        pass_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(n_pass)]
        # the stand-in compute alone, same launches, no library calls
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for l in range(N):
            torch.cuda._sleep(cycles)
            scratch.copy_(chunk)
        e1.record(stream)
        torch.cuda.synchronize(device)
        compute_ms = e0.elapsed_time(e1)
        st1 = lw.stats()
    finally:
        lw.close()
    h2d = (st1["bytes_h2d"] - st0["bytes_h2d"]) / n_pass
    d2h = (st1["bytes_d2h"] - st0["bytes_d2h"]) / n_pass
    t_pass = statistics.median(pass_ms)  # host-link transients of a shared node hit single passes
    t_h2d = h2d / (link["h2d"] * 1e9) * 1e3
    t_d2h = d2h / (link["d2h"] * 1e9) * 1e3
    t_roof = max(compute_ms, t_h2d, t_d2h)
    return {
        "layers": N, "trays": 4, "prefix_tokens": L0, "chunk_tokens": c, "passes": n_pass,
        "ms_per_pass": round(t_pass, 4), "ms_per_pass_mean": round(statistics.mean(pass_ms), 4),
        "pass_ms": [round(x, 3) for x in pass_ms], "compute_window_us_per_layer": round(win_us, 1),
        "compute_ms_per_pass": round(compute_ms, 4),
        "exposed_transfer_ms_per_pass": round(max(0.0, t_pass - compute_ms), 4),
        "h2d_bytes_per_pass": int(h2d), "d2h_bytes_per_pass": int(d2h),
        "h2d_gbs": round(h2d / (t_pass * 1e-3) / 1e9, 1), "d2h_gbs": round(d2h / (t_pass * 1e-3) / 1e9, 1),
        "roofline": {"bound": "compute window" if compute_ms >= max(t_h2d, t_d2h) else "host link",
                     "t_roofline_ms": round(t_roof, 4), "frac": round(t_roof / t_pass, 4),
                     "peaks_gbs": {"h2d": round(link["h2d"], 1), "d2h": round(link["d2h"], 1)}},
        "device_buffer_bytes": 4 * T * row * 2, "host_pool_bytes": N * T * row * 2,
        "host_pool_huge_backed": huge_frac, "host_pool_numa": pool_numa,
    }


# --------------------------------------------------------------------------- GPU arm
def run_kvo(args, log):
    import numpy as np
    import torch
    from top_cache_gb300 import kvo as K

    world, rank = dist_init("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    wl = make_workload(args)
    hbm_peak, hbm_src = load_peaks()
    link = measure_host_link(torch, device)
    kv, inp, units = prepare(wl, rank, device, log, args.idx, args.host_block_tokens)
    U, P, k, R = len(units), wl.n_pos, wl.topk, wl.row_elems
    kv.set_option(K.KVO_OPT_GATHER_MODE, K.KVO_GATHER_BULK if args.gather == "bulk" else K.KVO_GATHER_LDG)
    # options left unset keep the library's per-call choice
    if args.groups is not None:
        kv.set_option(K.KVO_OPT_GROUPS, args.groups)
    if args.score_ctas:
        kv.set_option(K.KVO_OPT_SCORE_CTAS, args.score_ctas)
    if args.group_gather_sms is not None:
        kv.set_option(K.KVO_OPT_GROUP_GATHER_SMS, args.group_gather_sms)
    if args.speculate is not None:
        kv.set_option(K.KVO_OPT_SPECULATE, args.speculate)
    if args.path != "auto":
        kv.set_option(K.KVO_OPT_FUSED, 1 if args.path == "fused" else 0)
    if args.path != "staged":
        if args.gather_ctas is not None:
            kv.set_option(K.KVO_OPT_GATHER_CTAS, args.gather_ctas)
        if args.piece_tokens is not None:
            kv.set_option(K.KVO_OPT_PIECE_TOKENS, args.piece_tokens)
    seq = Sequence(kv, inp, wl)
    stream = torch.cuda.current_stream(device)

    # the clock sampler starts before the warm-up, so that its start-up (nvidia-smi
    # initialising NVML) overlaps the warm-up steps rather than the timed ones
    sampler = ClockSampler(local)
    t_s = time.time()
    while not sampler.samples and time.time() - t_s < 5.0:
        time.sleep(0.05)
    # warm-up (the first step of the sequence is the cold, all-miss step)
    for _ in range(args.warmup):
        seq.step()
    torch.cuda.synchronize(device)
    kv.profile_read()
    # in the timed region only the kernels a roofline is reported for are bracketed with
    # events (each pair adds a few microseconds between launches); the small kernels'
    # times come from a replay of the same positions afterwards
    kv.set_option(K.KVO_OPT_PROFILE_KINDS, _kinds_mask(TIMED_KINDS))
    kv.set_option(K.KVO_OPT_PROFILE, 1)
    st0 = kv.stats()

    # ---------------- timed region
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    positions = []
    barrier(world)
    torch.cuda.synchronize(device)
    t_wall0 = time.time()
    ev[0].record(stream)
    for i in range(args.steps):
        positions.append(seq.step())
        ev[i + 1].record(stream)
    torch.cuda.synchronize(device)
    t_wall1 = time.time()
    barrier(world)
    step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    total_ms = ev[0].elapsed_time(ev[args.steps])
    prof = kv.profile_read()
    kv.set_option(K.KVO_OPT_PROFILE, 0)
    st1 = kv.stats()
    # keep the GPU busy a little longer so the clock sampler sees the load
    t_c0 = time.time()
    while time.time() - t_c0 < 1.0:
        seq.step()
        torch.cuda.synchronize(device)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)

    # replay of the timed positions with every launch bracketed (the small kernels' times)
    kv.reset(wl.context)
    seq = Sequence(kv, inp, wl)
    for _ in range(args.warmup):
        seq.step()
    torch.cuda.synchronize(device)
    kv.profile_read()
    kv.set_option(K.KVO_OPT_PROFILE_KINDS, (1 << len(K.PROF_KINDS)) - 1)
    kv.set_option(K.KVO_OPT_PROFILE, 1)
    for _ in range(args.steps):
        seq.step()
    torch.cuda.synchronize(device)
    prof_all = kv.profile_read()
    kv.set_option(K.KVO_OPT_PROFILE, 0)
    for name, (ms, n) in prof_all.items():
        if name not in TIMED_KINDS and n:
            prof[name] = (ms, n)

    # the cold step on its own: every unit back at its prefilled context with an empty
    # shelf, then step 0 of the sequence (every selected row a miss), three times
    cold_ms = []
    for _ in range(3):
        kv.reset(wl.context)
        seq = Sequence(kv, inp, wl)
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        c0.record(stream)
        seq.step()
        c1.record(stream)
        torch.cuda.synchronize(device)
        cold_ms.append(c0.elapsed_time(c1))

    fused_frac = (st1["fused_steps"] - st0["fused_steps"]) / args.steps
    path = "fused" if fused_frac == 1 else "staged" if fused_frac == 0 else "mixed (%.0f%% fused)" % (100 * fused_frac)
    split_frac = (st1["split_steps"] - st0["split_steps"]) / args.steps
    if split_frac == 1:
        path = "staged, two unit groups (the first group's rows copied inside the second's score launch)"
    elif split_frac > 0:
        path += " (%.0f%% in split unit groups)" % (100 * split_frac)
    max_ms = reduce_max(total_ms, world, device)
    value = whole_job_rate(U, args.steps, max_ms, world)

    # ---------------- per-kernel roofline
    rows_h2d = st1["rows_h2d"] - st0["rows_h2d"]
    bytes_h2d = st1["bytes_h2d"] - st0["bytes_h2d"]
    lens = [wl.context + (p + 1) * wl.n_new for p in positions]  # tokens per unit after append
    key_bytes = 130.0 if args.idx == "int8" else 256.0  # int8: code row + fp16 scale
    score_bytes = sum(key_bytes * U * L for L in lens)
    append_bytes = args.steps * U * wl.n_new * (R * 2 + 256)
    kernels = {}
    for name, (ms, n) in prof.items():
        if n == 0:
            continue
        kernels[name] = {"launches": n, "ms_total": round(ms, 4), "ms_per_launch": round(ms / n, 5),
                         "share": round(ms / max(1e-9, sum(v[0] for v in prof.values())), 4),
                         "timed": "in the timed region" if name in TIMED_KINDS
                                  else "replay of the timed positions"}
    # per-launch bytes: a step runs either the staged or the fused launches (with the
    # per-call choice both can appear in one run), and a staged step in unit groups runs
    # one score and one gather launch per group, each over its own units: the bytes of
    # all staged steps divided by their launches
    score_step = score_bytes / args.steps
    rows_step = bytes_h2d / args.steps
    n_fused = prof["fused"][1] if "fused" in prof else 0
    staged_steps = args.steps - n_fused
    if "score" in kernels and staged_steps:
        sb = score_step * staged_steps
        a = sb / (prof["score"][0] / 1e3) / 1e9
        if st1["rows_h2d_in_score"] > st0["rows_h2d_in_score"]:
            kernels["score"]["note"] = ("%.0f MB of miss rows per step copied by the first CTAs of "
                                        "the second group's score launch"
                                        % ((st1["rows_h2d_in_score"] - st0["rows_h2d_in_score"])
                                           * R * 2 / args.steps / 1e6))
        kernels["score"].update(bound="hbm", bytes_per_launch=sb / prof["score"][1],
                                achieved_gbs=round(a, 1), peak_gbs=hbm_peak,
                                frac=round(a / hbm_peak, 4), peak_source=hbm_src)
    # rows copied by the first CTAs of a score launch (staged step in unit groups) are
    # not the gather launches' bytes
    carried_b = (st1["rows_h2d_in_score"] - st0["rows_h2d_in_score"]) * R * 2
    if "gather" in kernels and bytes_h2d - carried_b > 0 and staged_steps:
        gb = (bytes_h2d - carried_b) / args.steps * staged_steps
        a = gb / (prof["gather"][0] / 1e3) / 1e9
        kernels["gather"].update(bound="host-link", bytes_per_launch=gb / prof["gather"][1],
                                 achieved_gbs=round(a, 1), peak_gbs=round(link["h2d"], 1),
                                 frac=round(a / link["h2d"], 4),
                                 peak_source="measured pinned host->device copy, this run")
    if "fused" in kernels:
        # one launch moves both the keys (HBM) and the miss rows (host link):
        # its bound is whichever takes longer at its peak
        t = prof["fused"][0] / 1e3
        nf = prof["fused"][1]
        rows_b = rows_step * nf
        hbm_b = (score_step + rows_step) * nf
        t_hbm, t_link = hbm_b / (hbm_peak * 1e9), rows_b / (link["h2d"] * 1e9)
        hbm_gbs, link_gbs = hbm_b / t / 1e9, rows_b / t / 1e9
        if t_link >= t_hbm:
            kernels["fused"].update(bound="host-link", achieved_gbs=round(link_gbs, 1),
                                    peak_gbs=round(link["h2d"], 1), frac=round(t_link / t, 4),
                                    peak_source="measured pinned host->device copy, this run")
        else:
            kernels["fused"].update(bound="hbm", achieved_gbs=round(hbm_gbs, 1), peak_gbs=hbm_peak,
                                    frac=round(t_hbm / t, 4), peak_source=hbm_src)
        kernels["fused"].update(bytes_per_launch=hbm_b / nf, hbm_gbs=round(hbm_gbs, 1),
                                host_link_gbs=round(link_gbs, 1),
                                hbm_frac=round(hbm_gbs / hbm_peak, 4),
                                host_link_frac=round(link_gbs / link["h2d"], 4))
    if "append" in kernels:
        a = append_bytes / (prof["append"][0] / 1e3) / 1e9
        kernels["append"].update(achieved_gbs=round(a, 1))
    for name in kernels:
        kernels[name]["traffic"] = load_traffic(name, wl.name)
    dom = max(kernels, key=lambda n: kernels[n]["ms_total"])
    d = kernels[dom]
    roof = {"kernel": dom, "bound": d.get("bound", "latency"),
            "achieved": d.get("achieved_gbs"), "peak": d.get("peak_gbs"), "unit": "GB/s",
            "frac": d.get("frac"), "traffic": load_traffic(dom, wl.name),
            "peak_source": d.get("peak_source")}

    # step roofline: slower of HBM bytes at peak and host-link bytes at measured bandwidth
    n_steps = args.steps
    hbm_step = (score_bytes + U * n_steps * (wl.n_new * 256 + 8 * wl.hot_capacity + 16 * P * k)
                + bytes_h2d) / n_steps
    host_step = (bytes_h2d + args.steps * U * wl.n_new * R * 2) / n_steps
    t_roof = max(hbm_step / (hbm_peak * 1e9), host_step / (link["h2d"] * 1e9)) * 1e3
    t_meas = total_ms / n_steps
    cold = [m for m, p in zip(step_ms, positions) if p == 0]
    warm = [m for m, p in zip(step_ms, positions) if p != 0]

    # ---------------- sparse attention over the hot buffer (decode step 7), timed on its own
    attention = None
    if args.attend_heads > 0 and wl.row_elems == 576:
        attention = run_attention(args, kv, wl, units, device, torch)
        attention["copy_sfa"] = run_copy_sfa(args, kv, inp, wl, units, device, torch)

    # ---------------- layerwise prefill offload, timed on its own
    layerwise = None
    if args.lw_layers > 0 and world == 1:
        layerwise = run_layerwise(args, link, device, torch, log)

    # ---------------- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, kv, inp, wl, U, device, world, torch)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = run_cpu_baseline(wl, args.cpu_units, min(args.cpu_steps, wl.steps), log)

    launches = st1["launches"] - st0["launches"]
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,1) bf16 keys and rows, random-walk queries)",
        "config": {"workload": wl.name, "n_requests": wl.n_requests, "n_layers": wl.n_layers,
                   "context": wl.context, "n_pos": P, "n_new": wl.n_new, "topk": k,
                   "hot_capacity": wl.hot_capacity, "drift": wl.drift,
                   "steps_per_sequence": wl.steps, "path": path, "indexer": args.idx,
                   "host_pool_page": kv.get_option(K.KVO_OPT_HOST_HUGE_PAGE) or "base",
                   "host_pool_huge_backed": huge_backed_fraction(
                       kv.host_block(0) if args.host_block_tokens else kv.host_rows(0)),
                   "host_pool_numa": numa_spread(
                       kv.host_block(0) if args.host_block_tokens else kv.host_rows(0)),
                   "gpu_numa_node": gpu_numa_node(device.index if device.index is not None else 0),
                   "host_block_tokens": args.host_block_tokens or None,
                   "gather": "bulk" if path == "fused" else args.gather, "groups": args.groups if args.groups is not None else "per call",
                   "parallelism": "replicas%d" % world,
                   "l2": "inputs larger than L2: %.2f GB of indexer keys read per step"
                         % (score_bytes / n_steps / 1e9)},
        "roofline": roof,
        "miss_fill": {"gbs": kernels.get("gather", kernels.get("fused", {})).get(
                          "achieved_gbs" if "gather" in kernels else "host_link_gbs"),
                      "peak_gbs": round(link["h2d"], 1), "rows_per_step": rows_h2d / n_steps,
                      "frac": kernels.get("gather", kernels.get("fused", {})).get(
                          "frac" if "gather" in kernels else "host_link_frac")},
        "step_roofline": {"hbm_bytes": round(hbm_step), "host_link_bytes": round(host_step),
                          "t_roofline_ms": round(t_roof, 4), "t_measured_ms": round(t_meas, 4),
                          "frac": round(t_roof / t_meas, 4)},
        "steps_ms": {"median": round(statistics.median(step_ms), 4),
                     "p90": round(sorted(step_ms)[int(0.9 * (len(step_ms) - 1))], 4),
                     "warm_median": round(statistics.median(warm), 4) if warm else None,
                     # the cold step: from the timed loop when it covered position 0, else
                     # the step 0 timed on its own after it
                     "cold_median": round(statistics.median(cold if cold else cold_ms), 4),
                     "cold_step_alone_ms": round(statistics.median(cold_ms), 4),
                     "p99": round(sorted(step_ms)[int(0.99 * (len(step_ms) - 1))], 4),
                     "max": round(max(step_ms), 4),
                     # the slowest steps as (position in the sequence, ms): tells a slow
                     # cold start from stalls that hit arbitrary steps
                     "slowest": [(positions[i], round(step_ms[i], 3)) for i in
                                 sorted(range(len(step_ms)), key=lambda i: -step_ms[i])[:8]]},
        "kernels": kernels,
        "host_link_gbs": {k_: round(v, 1) for k_, v in link.items()},
        "hits_per_step": (st1["hits"] - st0["hits"]) / n_steps,
        "misses_per_step": (st1["misses"] - st0["misses"]) / n_steps,
        "rescored_units_per_step": (st1["rescored"] - st0["rescored"]) / n_steps,
        "clocks": clocks,
        "e2e": e2e,
        "attention": attention,
        "layerwise_prefill": layerwise,
        "gpu_launches": launches,
        "cpu_baseline": cpu,
    }
    kv.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(args, kv, inp, wl, U, device, world, torch):
    """Same steps through the public API with pinned host inputs and outputs.

    Every step copies its inputs host -> device before the step and its
    outputs (tokens, slots, scores, status) device -> host after it, all inside
    the timed region.  As a serving loop would, the read-back of step s runs on
    a copy stream while step s+1 computes (outputs double-buffered; the host
    reads step s's status once its copy has landed)."""
    P, k = wl.n_pos, wl.topk
    pin = lambda a: torch.from_numpy(a).pin_memory()
    rows_h, keys_h, q_h = pin(inp["rows_h"]), pin(inp["keys_h"]), pin(inp["q_h"])
    rows_d = torch.empty_like(inp["rows"][0])
    keys_d = torch.empty_like(inp["keys"][0])
    q_d = torch.empty_like(inp["q"][0])

    def outputs():
        return (torch.empty((U, P, k), dtype=torch.int32, device=device),
                torch.empty((U, P, k), dtype=torch.int32, device=device),
                torch.empty((U, P, k), dtype=torch.float32, device=device),
                torch.empty((U, P, k), dtype=torch.int32, device=device),
                torch.empty(U, dtype=torch.int32, device=device))

    out_d = [outputs(), outputs()]
    out_h = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in o] for o in out_d]
    read = (0, 1, 2, 4)  # tokens, slots, scores, status come back every step
    main = torch.cuda.current_stream(device)
    copy = torch.cuda.Stream(device)
    done = [torch.cuda.Event(), torch.cuda.Event()]
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    kv.reset(wl.context)
    g = 0
    n = args.steps
    h2d = (rows_d.numel() + keys_d.numel() + q_d.numel()) * 2
    d2h = sum(out_d[0][i].numel() * out_d[0][i].element_size() for i in read)
    bad = 0
    for warm in (True, False):
        steps = min(args.warmup, n) if warm else n
        barrier(world)
        torch.cuda.synchronize(device)
        t0 = time.perf_counter()
        for j in range(steps):
            p = g % wl.steps
            b = g % 2
            if j >= 2:
                main.wait_event(copied[b])  # outputs b free again
            if p == 0 and g > 0:
                kv.reset(wl.context)
            rows_d.copy_(rows_h[p], non_blocking=True)
            keys_d.copy_(keys_h[p], non_blocking=True)
            q_d.copy_(q_h[p], non_blocking=True)
            kv.append(rows_d, keys_d)
            kv.step(q_d, out=out_d[b])
            done[b].record(main)
            copy.wait_event(done[b])
            with torch.cuda.stream(copy):
                for i in read:
                    out_h[b][i].copy_(out_d[b][i], non_blocking=True)
            copied[b].record(copy)
            if j >= 1:
                copied[1 - b].synchronize()
                bad += int((out_h[1 - b][4] != 0).sum())
            g += 1
        copied[(g - 1) % 2].synchronize()
        bad += int((out_h[(g - 1) % 2][4] != 0).sum())
        t1 = time.perf_counter()
    ms = reduce_max((t1 - t0) * 1e3, world, device)
    return {"value": round(whole_job_rate(U, n, ms, world), 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms / n, 4), "units_not_ok": bad,
            "pipelining": "read-back of step s overlaps step s+1 (copy stream, double-buffered outputs)"}


# --------------------------------------------------------------------------- CPU oracle
def run_cpu_baseline(wl, n_units, n_steps, log, units_offset=0, max_seconds=30.0):
    """The CPU oracle, as it stands, on a bounded sample of the same workload: n_units units
    over up to n_steps steps of the sequence, stopping early once the warm steps have taken
    max_seconds."""
    import numpy as np
    import oracle
    import workload as W

    units = wl.units_rl()[units_offset:units_offset + n_units]
    tmax = wl.max_tokens(n_steps)
    keys = W.token_rows(wl.seed, W.KIND_KEYS, units, 0, tmax, 128)
    rows = W.token_rows(wl.seed, W.KIND_ROWS, units, 0, tmax, wl.row_elems)
    q = W.unit_queries(wl.seed, units, wl.drift, n_steps, wl.n_pos)
    ors = []
    for i in range(len(units)):
        o = oracle.OracleUnit(tmax, wl.topk, wl.hot_capacity, wl.n_pos, wl.row_elems, keep_rows=True)
        o.append(keys[i, :wl.context], rows[i, :wl.context])
        ors.append(o)
    timed = 0.0
    L = wl.context
    done = 0
    for s in range(n_steps):
        t0 = time.perf_counter()
        for i, o in enumerate(ors):
            o.append(keys[i, L:L + wl.n_new], rows[i, L:L + wl.n_new])
        oracle.step_many(ors, q[s])
        dt = time.perf_counter() - t0
        L += wl.n_new
        done = s + 1
        if s > 0:
            timed += dt
            if timed >= max_seconds:
                break
    n = len(units) * (done - 1)
    log("cpu oracle: %d unit-steps in %.2f s" % (n, timed))
    return {"value": round(n / timed, 2), "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
            "sample": "%d of %d units (%s), %d warm steps after one cold step, context %d"
                      % (len(units), wl.n_units, wl.name, done - 1, wl.context)}


def run_reference(args, log):
    """Reference arm: the CPU oracle timed on this machine's host cores."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np
    import oracle
    import workload as W

    wl = make_workload(args)
    # size the per-step sample so that the whole run ends within a few minutes
    probe = run_cpu_baseline(wl, min(16, wl.n_units), 2, log)
    per_unit_s = 1.0 / probe["value"]
    budget_s = 90.0
    n_units = int(max(1, min(wl.n_units, budget_s / max(1, args.steps + args.warmup) / per_unit_s)))
    # Units are independent, so a sample of a few units per core measures the same rate;
    # the cap also bounds the untimed set-up (generating and loading each unit's prefill
    # rows, 38 MB per unit on batch16x8_32k_mtp3), which otherwise dominates the run.
    n_units = min(n_units, max(32, 2 * oracle.threads()))
    units = wl.units_rl()[:n_units]
    S = wl.steps
    tmax = wl.max_tokens(S)
    keys = W.token_rows(wl.seed, W.KIND_KEYS, units, 0, tmax, 128)
    rows = W.token_rows(wl.seed, W.KIND_ROWS, units, 0, tmax, wl.row_elems)
    q = W.unit_queries(wl.seed, units, wl.drift, S, wl.n_pos)

    def fresh():
        ors = []
        for i in range(n_units):
            o = oracle.OracleUnit(tmax, wl.topk, wl.hot_capacity, wl.n_pos, wl.row_elems, True)
            o.append(keys[i, :wl.context], rows[i, :wl.context])
            ors.append(o)
        return ors

    ors = fresh()
    g = 0
    timed = 0.0
    for i in range(args.warmup + args.steps):
        p = g % S
        if p == 0 and g > 0:
            ors = fresh()  # the sequence starts again from the prefill (untimed)
        L = wl.context + p * wl.n_new
        t0 = time.perf_counter()
        for j, o in enumerate(ors):
            o.append(keys[j, L:L + wl.n_new], rows[j, L:L + wl.n_new])
        oracle.step_many(ors, q[p])
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            timed += dt
        g += 1
    value = n_units * args.steps / timed
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(timed * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,1) bf16 keys and rows, random-walk queries)",
        "config": {"workload": wl.name, "n_requests": wl.n_requests, "n_layers": wl.n_layers,
                   "context": wl.context, "n_pos": wl.n_pos, "n_new": wl.n_new,
                   "topk": wl.topk, "hot_capacity": wl.hot_capacity, "drift": wl.drift,
                   "steps_per_sequence": S, "parallelism": "replicas%d" % world},
        "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": oracle.threads(),
                         "kind": "oracle",
                         "sample": "%d of %d units per step (%s), context %d"
                                   % (n_units, wl.n_units, wl.name, wl.context)},
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("kvo", "reference"), default="kvo")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--requests", type=int, default=0)
    ap.add_argument("--layers", type=int, default=0)
    ap.add_argument("--context", type=int, default=0)
    ap.add_argument("--drift", type=float, default=None,
                    help="query drift a of the workload (the sweep workload's points: 0, .5, .9, .99, 1)")
    ap.add_argument("--gather", choices=("ldg", "bulk"), default="ldg")
    ap.add_argument("--groups", type=int, default=None,
                    help="unit groups per step; miss-row copies overlap the next group's scoring")
    ap.add_argument("--score-ctas", type=int, default=0, help="cap on scoring CTAs (0 = one per SM)")
    ap.add_argument("--group-gather-sms", type=int, default=None,
                    help="staged step in unit groups: CTAs of each score launch that copy the previous group's rows")
    ap.add_argument("--path", choices=("auto", "fused", "staged"), default="auto",
                    help="fused: one cooperative launch per step; staged: one launch per stage; "
                         "auto: the library's default for the configuration")
    ap.add_argument("--gather-ctas", type=int, default=None, help="fused step: CTAs that only fill rows")
    ap.add_argument("--idx", choices=("bf16", "int8"), default="bf16",
                    help="indexer cache format (int8: Hadamard-rotated int8 codes + fp16 scales)")
    ap.add_argument("--speculate", type=int, default=None,
                    help="speculative threshold margin in permille (library default 900)")
    ap.add_argument("--piece-tokens", type=int, default=None, help="fused step: tokens per piece")
    ap.add_argument("--attend-heads", type=int, default=128,
                    help="heads of the timed sparse attention (multiple of 128; 0 = skip it)")
    ap.add_argument("--attend-launches", type=int, default=20)
    ap.add_argument("--lw-layers", type=int, default=78,
                    help="layers of the timed layerwise prefill passes (0 = skip them)")
    ap.add_argument("--lw-prefix", type=int, default=16384)
    ap.add_argument("--lw-chunk", type=int, default=4096)
    ap.add_argument("--lw-passes", type=int, default=5)
    ap.add_argument("--lw-window-us", type=float, default=0.0,
                    help="stand-in compute per layer (0 = the layer's load time at the measured peak)")
    ap.add_argument("--host-block-tokens", type=int, default=0,
                    help="paged host pool: rows per block, blocks scattered by a seeded permutation (0 = per-unit rows)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-units", type=int, default=32)
    ap.add_argument("--cpu-steps", type=int, default=50)  # at most the sequence's own steps
    ap.add_argument("--quiet", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    log = (lambda *a: None) if args.quiet else (lambda m: print("[bench] " + m, file=sys.stderr, flush=True))
    if args.impl == "reference":
        run_reference(args, log)
    else:
        import __graft_entry__
        __graft_entry__.build()
        run_kvo(args, log)


if __name__ == "__main__":
    main()
