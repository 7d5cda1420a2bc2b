"""Benchmark: causal GQA attention forward + backward on GB300.

One step = one forward (attn_fwd) and one backward (attn_bwd) of the long
context GQA layer (B=2, Hq=32, Hkv=8, T=4096, D=128, causal, bf16) over one
batch of synthetic inputs already resident in HBM.  The L2 cache (129 MB) is
evicted before every timed step by reading a 256 MiB buffer (clean lines:
nothing is written back during the step; --flush write writes it instead);
the step itself is timed
with CUDA events on the launching stream.  FLOPs follow the causal convention
(half of dense): forward 4*D and backward 10*D per visible (query, key) pair,
i.e. 2*B*Hq*T^2*D and 5*B*Hq*T^2*D.

Before the timed steps, one forward + backward is compared with the fp64
oracle (the whole workload, or one sampled (batch, kv-head) group of the
long-context layer) and the figures go into the line's "parity" object.
Per-kernel times come from a second pass of as many steps with CUDA events
around every kernel, so the timed steps carry none.

Prints one JSON line.  --impl reference times the fp64 CPU oracle (the only
reference this method has) on a bounded sample of the same workload.

--workload decode_* measures cached (decode) attention instead: one step is
one attn_decode_fwd call over a KV cache resident in HBM (larger than L2 for
the long-context workload, and L2 is evicted before every step anyway); the
figure is algorithmic HBM bytes per second -- the K and V rows each batch
row actually holds (cache_lens[b] keys, Hkv heads, D features, bf16) plus Q,
O, LSE and the lengths -- against the measured copy bandwidth.
Multi-GPU: each rank runs an independent replica (the path has no exchange
step); value = all ranks' FLOPs / max over ranks of the timed region.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from causal_gqa_attention_fwd_gb300 import workloads as W  # noqa: E402

METRIC = "causal GQA attention fwd+bwd TFLOP/s (bf16) and % of GB300 tensor peak"


class L2Flush:
    """Evicts the L2 cache (129 MB) between timed steps with a 256 MiB buffer:
    'read' reads it (the evicted lines are clean, so nothing is written back
    while the next step runs), 'write' writes it (its dirty lines are then
    written back to HBM during the next step), 'none' does nothing."""

    def __init__(self, mode: str, dev):
        self.mode = mode
        self.buf = None if mode == "none" else torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.sink = None

    def __call__(self, i: int = 0):
        if self.mode == "read":
            self.sink = torch.amax(self.buf)
        elif self.mode == "write":
            self.buf.fill_(i & 0xFF)

    def describe(self) -> str:
        return {"read": "evicted before every timed step by reading a 256 MiB buffer",
                "write": "flushed before every timed step by writing a 256 MiB buffer",
                "none": "not flushed"}[self.mode]

UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 256 << 20


def flops(w: W.Workload, cu=None):
    """(fwd, bwd) algorithmic FLOPs, causal counted as half of dense."""
    if w.varlen:
        lens = (cu[1:] - cu[:-1]).to(torch.int64)
        sq = int((lens * lens).sum())
    else:
        sq = w.B * w.T * w.T
    pairs = w.Hq * sq / (2.0 if w.causal else 1.0)
    return 4.0 * w.D * pairs, 10.0 * w.D * pairs


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"bf16_tflops": d["bf16_tflops"], "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


def measured_traffic(workload: str, kernel: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum)
    from the committed ncu capture, or None if there is none for this
    workload or the kernel's sources changed since it was taken."""
    import hashlib
    tp = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(tp):
        return None
    entry = json.load(open(tp)).get(workload, {}).get(kernel)
    if not entry:
        return None
    h = hashlib.sha256()
    for f in entry["sources"]:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return entry["dram_bytes_per_launch"] if h.hexdigest()[:16] == entry["source_sha256_16"] else None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == 0:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for t, line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                rows.append((t, float(f[2]), float(f[3]), f[5:10]))
            except ValueError:
                continue
        if not rows:
            return None
        inside = [r for r in rows if self.t0 - 0.15 <= r[0] <= self.t1 + 0.15] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3][1:]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


# ------------------------------------------------------------- CPU oracle
def oracle_sample(w: W.Workload, x, budget_s: float, t_prefix: int | None = None):
    """Time the fp64 oracle on whole (batch, kv-head) groups of the workload
    (packed batches: whole sequences, every head) until about budget_s
    seconds of CPU work (at least one group).  With t_prefix, each group is
    cut to its first t_prefix positions (a causal prefix is itself a complete
    causal problem).  Returns (FLOP/s, sample description, cores, seconds)."""
    import numpy as np

    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    if w.varlen:
        f = lambda t: t.float().numpy().astype(np.float64)
        cu = x["cu_seqlens"].tolist()
        nseq = len(cu) - 1
        done_flops, elapsed, seqs = 0.0, 0.0, 0
        while seqs == 0 or (elapsed < budget_s and seqs < nseq):
            a, b = cu[seqs], cu[seqs + 1]
            sub_cu = np.array([0, b - a], dtype=np.int32)
            q, k, v, do = (f(x[n][a:b]) for n in ("q", "k", "v", "do"))
            t0 = time.perf_counter()
            oracle.varlen_bwd(q, k, v, do, sub_cu, causal=w.causal, scale=w.softmax_scale)  # forward + backward
            elapsed += time.perf_counter() - t0
            seqs += 1
            ff, fb = flops(W.Workload("s", B=1, Hq=w.Hq, Hkv=w.Hkv, T=b - a, D=w.D, causal=w.causal))
            done_flops += ff + fb
        desc = (f"the first {seqs} of {nseq} packed sequences of {w.name} (lengths {[cu[i + 1] - cu[i] for i in range(seqs)]}), "
                f"every head, forward + backward in fp64, {elapsed:.1f} s")
        return done_flops / elapsed, desc, cores, elapsed
    G = w.Hq // w.Hkv
    T = min(w.T, t_prefix) if t_prefix else w.T
    done_flops, elapsed, groups = 0.0, 0.0, 0
    f = lambda t: t.float().numpy().astype(np.float64)
    total_groups = w.B * w.Hkv
    while groups == 0 or (elapsed < budget_s and groups < total_groups):
        b, g = divmod(groups, w.Hkv)
        q = f(x["q"][b:b + 1, g * G:(g + 1) * G, :T])
        k = f(x["k"][b:b + 1, g:g + 1, :T])
        v = f(x["v"][b:b + 1, g:g + 1, :T])
        do = f(x["do"][b:b + 1, g * G:(g + 1) * G, :T])
        t0 = time.perf_counter()
        oracle.bwd(q, k, v, do, causal=w.causal, scale=w.softmax_scale)   # forward + backward
        elapsed += time.perf_counter() - t0
        groups += 1
        ff, fb = flops(W.Workload("s", B=1, Hq=G, Hkv=1, T=T, D=w.D, causal=w.causal))
        done_flops += ff + fb
    where = f"first {T} of T={w.T} positions" if T < w.T else f"full T={w.T}"
    desc = (f"{groups} of {total_groups} (batch, kv-head) groups of {w.name}, {where} "
            f"(G={G} query heads each), forward + backward in fp64, {elapsed:.1f} s")
    return done_flops / elapsed, desc, cores, elapsed


# ------------------------------------------------------------- parity leg
def parity_leg(w: W.Workload, x, out: dict):
    """Compare one forward + backward of the GPU path with the fp64 oracle,
    outside the timed region: the whole workload, or for the long-context
    layer one sampled (batch, kv-head) group (every row of its G query heads
    and of its K/V head).  Returns every figure of ``oracle.parity`` per
    output and which elementwise bound it meets."""
    import numpy as np

    import oracle
    from oracle import parity as P
    oracle.build()
    oracle.set_threads(len(os.sched_getaffinity(0)))
    f = lambda t: t.detach().float().cpu().numpy().astype(np.float64)
    t0 = time.perf_counter()
    G = w.Hq // w.Hkv
    if w.varlen:
        # the shortest and the longest packed sequence (sequences are independent)
        cu = x["cu_seqlens"].tolist()
        lens = [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]
        pick = sorted({min(range(len(lens)), key=lambda i: lens[i]), max(range(len(lens)), key=lambda i: lens[i])})
        rows = torch.cat([torch.arange(cu[i], cu[i + 1]) for i in pick])
        sub_cu = np.cumsum([0] + [lens[i] for i in pick]).astype(np.int32)
        ref = oracle.varlen_bwd(f(x["q"][rows]), f(x["k"][rows]), f(x["v"][rows]), f(x["do"][rows]), sub_cu,
                                causal=w.causal, scale=w.softmax_scale, err_terms=True)
        got = {n: f(out[n].cpu()[rows]) for n in ("o", "dq", "dk", "dv")}
        got["lse"] = f(out["lse"].cpu()[:, rows])
        sample = (f"packed sequences {pick} of {len(lens)} (lengths {[lens[i] for i in pick]}: the shortest and "
                  f"the longest), every head, forward and backward")
    elif w.B * w.T > 4096:
        b, g = 1, min(5, w.Hkv - 1)
        hs = slice(g * G, (g + 1) * G)
        ref = oracle.bwd(f(x["q"][b:b + 1, hs]), f(x["k"][b:b + 1, g:g + 1]), f(x["v"][b:b + 1, g:g + 1]),
                         f(x["do"][b:b + 1, hs]), causal=w.causal, scale=w.softmax_scale, err_terms=True)
        got = {n: f(out[n][b:b + 1, hs]) for n in ("o", "lse", "dq")}
        got.update({n: f(out[n][b:b + 1, g:g + 1]) for n in ("dk", "dv")})
        sample = f"(batch {b}, kv-head {g}) group: {G} query heads x {w.T} rows, forward and backward"
    else:
        ref = oracle.bwd(f(x["q"]), f(x["k"]), f(x["v"]), f(x["do"]), causal=w.causal, scale=w.softmax_scale,
                         err_terms=True)
        got = {n: f(out[n]) for n in ("o", "lse", "dq", "dk", "dv")}
        sample = "whole workload"
    res = {"o": P.compare("o", got["o"], ref["o"], P.TOL_REL_O)}
    for n in ("dq", "dk", "dv"):
        res[n] = P.compare(n, got[n], ref[n], P.TOL_REL_GRAD, ref["e" + n])
    lse = P.compare_lse(got["lse"], ref["lse"])
    keep = ("rel_fro", "rel_tol", "max_abs", "flat_excess", "ulp_excess", "widened_excess", "max_ref", "meets")
    outputs = {n: {k: r[k] for k in keep} for n, r in res.items()}
    outputs["lse"] = {"max_abs": lse["max_abs"], "tol": lse["tol"]}
    return {"against": "fp64 CPU oracle", "sample": sample,
            "tolerances": {"rel_fro_o": P.TOL_REL_O, "rel_fro_grad": P.TOL_REL_GRAD, "abs_flat": P.TOL_ABS,
                           "lse_abs": P.TOL_LSE,
                           "abs_widened": "2e-2 + bf16 half-ulp of ref (+ 3 * 2^-8 * e for dq/dk/dv)"},
            "outputs": outputs,
            "pass": all(r["ok"] for r in res.values()) and lse["ok"],
            "flat_pass": all(r["meets"] == "flat" for r in res.values()) and lse["ok"],
            "half_ulp_pass": all(r["meets"] in ("flat", "half-ulp") for r in res.values()) and lse["ok"],
            "seconds": time.perf_counter() - t0}


def decode_parity_leg(w, x, o, lse):
    """Compare one decode call with the fp64 oracle on two batch rows (the
    shortest and the longest cache; rows are independent), every head and
    query position.  Paged caches: only the pages those rows use are handed
    to the oracle, with the block table renumbered.  Returns O's figures of
    ``oracle.parity`` and the LSE error, as the prefill leg does."""
    import numpy as np

    import oracle
    from oracle import parity as P
    oracle.build()
    oracle.set_threads(len(os.sched_getaffinity(0)))
    t0 = time.perf_counter()
    f = lambda t: t.float().numpy().astype(np.float64)
    lens = x["cache_lens"]
    rows = sorted({int(lens.argmin()), int(lens.argmax())})
    q, ln = f(x["q"][rows]), lens[rows].numpy()
    rope = x["rope_cs"].double().numpy() if w.rope else None
    if w.fp8:
        ro, rlse = oracle.fp8_decode_fwd(q, x["k8"][rows].numpy(), x["v8"][rows].numpy(), x["k_scale"], x["v_scale"],
                                         ln, scale=w.softmax_scale, rope_cos_sin=rope)
    elif w.page_size:
        bt = x["block_table"][rows]
        used = sorted({int(e) for r, n in zip(bt, ln) for e in r[: (int(n) + w.page_size - 1) // w.page_size]})
        remap = {e: i for i, e in enumerate(used)}
        bt_sub = np.array([[remap.get(int(e), 0) for e in r] for r in bt], dtype=np.int32)
        idx = torch.tensor(used, dtype=torch.int64)
        ro, rlse = oracle.paged_decode_fwd(q, f(x["k_pages"][idx]), f(x["v_pages"][idx]), bt_sub, ln,
                                           scale=w.softmax_scale, rope_cos_sin=rope)
    else:
        ro, rlse = oracle.decode_fwd(q, f(x["k_cache"][rows]), f(x["v_cache"][rows]), ln, scale=w.softmax_scale,
                                     rope_cos_sin=rope)
    res = P.compare("o", f(o.cpu()[rows]), ro, P.TOL_REL_O)
    le = P.compare_lse(f(lse.cpu()[rows]), rlse)
    keep = ("rel_fro", "rel_tol", "max_abs", "flat_excess", "ulp_excess", "widened_excess", "max_ref", "meets")
    return {"against": "fp64 CPU oracle",
            "sample": f"batch rows {rows} (cache lengths {[int(v) for v in ln]}: the shortest and the longest), "
                      f"every head and query position",
            "tolerances": {"rel_fro_o": P.TOL_REL_O, "abs_flat": P.TOL_ABS, "lse_abs": P.TOL_LSE},
            "outputs": {"o": {k: res[k] for k in keep}, "lse": {"max_abs": le["max_abs"], "tol": le["tol"]}},
            "pass": res["ok"] and le["ok"], "flat_pass": res["meets"] == "flat" and le["ok"],
            "seconds": time.perf_counter() - t0}


def graph_launch_floor_us(stream, reps: int = 50) -> float:
    """Median time of replaying a CUDA graph of two minimal kernels (one-element
    writes): the launch floor under any two-kernel call such as a decode
    (partial + merge)."""
    t = torch.zeros(1, device="cuda")
    with torch.cuda.stream(stream):
        t.add_(1.0)
        t.add_(1.0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        t.add_(1.0)
        t.add_(1.0)
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        ts.append((a, b))
    torch.cuda.synchronize()
    ms = sorted(a.elapsed_time(b) for a, b in ts)
    return ms[len(ms) // 2] * 1e3


# ---------------------------------------------------------------- decode
DECODE_METRIC = "cached GQA decode attention: algorithmic HBM GB/s and % of GB300 copy bandwidth"
DECODE_UNIT = "GB/s"


def decode_bytes(w: W.DecodeWorkload, lens) -> int:
    """Algorithmic bytes of one decode call: K and V rows inside each row's
    cache (2 bytes each, 1 for E4M3 caches), Q read, O written (bf16), LSE
    written (f32), the lengths (paged: and the block-table entries of the
    pages that hold keys; rotary queries: the f32 table row of each query
    position)."""
    lens = torch.as_tensor(lens, dtype=torch.int64)
    kv = 2 * w.Hkv * w.D * (1 if w.fp8 else 2) * int(lens.sum())
    qo = 2 * w.B * w.Hq * w.Tq * w.D * 2
    table = 4 * int(((lens + w.page_size - 1) // w.page_size).sum()) if w.page_size else 0
    rope = 4 * w.D * w.B * w.Tq if w.rope else 0
    return kv + qo + w.B * w.Hq * w.Tq * 4 + w.B * 4 + table + rope


def oracle_decode_sample(w: W.DecodeWorkload, x, budget_s: float):
    """Time the fp64 oracle on whole batch rows of a decode workload until
    about budget_s seconds (at least one row).  Returns (bytes/s, sample
    description, cores, seconds)."""
    import numpy as np

    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    f = lambda t: t.float().numpy().astype(np.float64)
    done, elapsed, rows = 0, 0.0, 0
    kp = vp = None
    if w.page_size:
        kp, vp = f(x["k_pages"]), f(x["v_pages"])
    rope = x["rope_cs"].double().numpy() if w.rope else None
    while rows == 0 or (elapsed < budget_s and rows < w.B):
        b = rows
        lens = x["cache_lens"][b:b + 1]
        if w.fp8:
            args = (f(x["q"][b:b + 1]), x["k8"][b:b + 1].numpy(), x["v8"][b:b + 1].numpy(), x["k_scale"],
                    x["v_scale"], lens.numpy())
            fn = oracle.fp8_decode_fwd
        elif w.page_size:
            args = (f(x["q"][b:b + 1]), kp, vp, x["block_table"][b:b + 1].numpy(), lens.numpy())
            fn = oracle.paged_decode_fwd
        else:
            args = (f(x["q"][b:b + 1]), f(x["k_cache"][b:b + 1]), f(x["v_cache"][b:b + 1]), lens.numpy())
            fn = oracle.decode_fwd
        t0 = time.perf_counter()
        fn(*args, scale=w.softmax_scale, rope_cos_sin=rope)
        elapsed += time.perf_counter() - t0
        rows += 1
        one = W.DecodeWorkload("s", B=1, Hq=w.Hq, Hkv=w.Hkv, Tq=w.Tq, S=w.S, D=w.D, min_len=0, max_len=0,
                               page_size=w.page_size, fp8=w.fp8, rope=w.rope)
        done += decode_bytes(one, lens)
    desc = f"{rows} of {w.B} batch rows of {w.name} (whole caches), fp64, {elapsed:.1f} s"
    return done / elapsed, desc, cores, elapsed


def decode_config(w: W.DecodeWorkload, world: int, l2: str):
    c = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Tq": w.Tq, "S": w.S, "D": w.D,
         "cache_lens": f"uniform in [{w.min_len}, {w.max_len}]",
         "parallelism": f"replicas x{world}" if world > 1 else "single GPU", "l2": l2}
    if w.page_size:
        c["paged"] = f"pages of {w.page_size} positions, [num_pages, Hkv, page, D], shuffled over the pool"
    if w.fp8:
        c["kv_cache"] = "E4M3 codes with one scale per cache (amax -> 448), N(0,1) source values"
    if w.rope:
        c["rope"] = "queries rotated in the kernel at their positions (rotate-half, base 10000, f32 table)"
    return c


def run_decode(args, world, rank, local):
    import causal_gqa_attention_fwd_gb300 as gq
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.DECODE_WORKLOADS[args.workload]
    x = W.make_decode_inputs(w, seed=rank)
    stream = torch.cuda.current_stream()
    if w.fp8:
        names = ("q", "k8", "v8", "cache_lens")
    elif w.page_size:
        names = ("q", "k_pages", "v_pages", "block_table", "cache_lens")
    else:
        names = ("q", "k_cache", "v_cache", "cache_lens")
    if w.rope:
        names = names + ("rope_cs",)
    dx = {n: x[n].to(dev) for n in names}
    q, lens = dx["q"], dx["cache_lens"]
    rcs = dx.get("rope_cs")
    scale = w.softmax_scale
    ws_bytes = gq.attn_decode_workspace_size(w.B, w.Hq, w.Hkv, w.Tq, w.S, w.D)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Tq), dtype=torch.float32, device=dev)

    def step():
        if w.fp8:
            gq.attn_decode_fp8_fwd(q, dx["k8"], dx["v8"], x["k_scale"], x["v_scale"], lens, scale=scale, o=o,
                                   lse=lse, workspace=ws, rope_cos_sin=rcs)
        elif w.page_size:
            gq.attn_decode_paged_fwd(q, dx["k_pages"], dx["v_pages"], dx["block_table"], lens, scale=scale, o=o,
                                     lse=lse, workspace=ws, rope_cos_sin=rcs)
        else:
            gq.attn_decode_fwd(q, dx["k_cache"], dx["v_cache"], lens, scale=scale, o=o, lse=lse, workspace=ws,
                               rope_cos_sin=rcs)

    step()

    # A decode step is a few microseconds of launches around a short kernel:
    # the timed steps replay the call captured in a CUDA graph (the call
    # allocates nothing and never synchronises), as a serving loop would.
    graph = None
    if not args.no_graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize()
    run = graph.replay if graph is not None else step

    nbytes = decode_bytes(w, x["cache_lens"])
    flush = L2Flush(args.flush, dev)
    for _ in range(args.warmup):
        flush(1)
        run()
    torch.cuda.synchronize()
    assert gq.get_device_status() == 0, "device status after warm-up"

    parity = None
    if rank == 0 and not args.no_parity:
        parity = decode_parity_leg(w, x, o, lse)
    floor_us = graph_launch_floor_us(stream)

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark(0)
    for i in range(args.steps):
        flush(i)
        ev[i][0].record(stream)
        run()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks.mark(1)
    # kernel-level events in a second pass of as many steps: an event recorded
    # between the partial and the merge kernel would stop the merge's
    # programmatic early launch, so the timed pass above records none
    gq.profile_reset()
    gq.profile_enable(True)
    for i in range(args.steps):
        flush(i)
        step()
    torch.cuda.synchronize()
    gq.profile_enable(False)
    prof = gq.profile_read()
    clk = clocks.stop()
    status = gq.get_device_status()
    total_ms = max_over_ranks(world, sum(a.elapsed_time(b) for a, b in ev))
    ms_per_step = total_ms / args.steps
    value = world * nbytes * args.steps / (total_ms / 1e3) / 1e9
    pk = peaks()
    n_part, t_part = prof["decode"]
    part_ms = t_part / max(n_part, 1)
    achieved = nbytes / (part_ms / 1e3) / 1e9
    roofline = {"kernel": "decode_partial", "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / pk["hbm_gbs"], "traffic": measured_traffic(w.name, "decode"),
                "peak_source": pk["source"] + " (copy bandwidth)", "algorithmic_bytes_per_launch": nbytes}

    e2e = None
    if not args.no_e2e:
        hx = {n: x[n].pin_memory() for n in names}
        ho, hlse = torch.empty_like(hx["q"]).pin_memory(), torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in hx.values())
        d2h = sum(t.numel() * t.element_size() for t in (ho, hlse))

        def e2e_step():
            for n in names:
                dx[n].copy_(hx[n], non_blocking=True)
            step()
            ho.copy_(o, non_blocking=True)
            hlse.copy_(lse, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        n_e2e = max(3, min(args.steps, 10))
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        torch.cuda.synchronize()
        e2e_s = max_over_ranks(world, time.perf_counter() - t0)
        e2e = {"value": world * nbytes * n_e2e / e2e_s / 1e9, "unit": DECODE_UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "note": "the whole KV cache crosses host->device every step"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, desc, cores, el = oracle_decode_sample(w, x, args.cpu_budget)
        cpu = {"value": rate / 1e9, "unit": DECODE_UNIT, "cores": cores, "kind": "oracle", "sample": desc}

    if rank == 0:
        line = {
            "metric": DECODE_METRIC, "value": value, "unit": DECODE_UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "data": "synthetic",
            "dtype": ("E4M3 K/V, bf16 q: scores E4M3 K x 3-part E4M3 q, P V f16 V x f16 P, f32 accumulation"
                      if w.fp8 else "bf16 in, f32 arithmetic"),
            "config": decode_config(w, world, flush.describe()),
            "frac_of_peak": value / pk["hbm_gbs"],
            "tokens_per_s": world * w.B * w.Tq * args.steps / (total_ms / 1e3),
            "kernel_ms": {k: (t / n if n else None) for k, (n, t) in prof.items() if n},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "parity": parity,
            "launch_floor_us": floor_us,
            "launch_floor": "median replay of a CUDA graph of two one-element kernels (a decode call launches two)",
            "gpu_launches": sum(prof[k][0] for k in prof), "kernel_ms_pass": "second pass, same steps, events per kernel",
            "launch": "CUDA graph replay of the call" if graph is not None else "eager calls",
            "clocks": clk, "device_status": status,
        }
        print(json.dumps(line), flush=True)


def run_decode_reference(args, world, rank):
    if rank != 0:
        return
    w = W.DECODE_WORKLOADS[args.workload]
    x = W.make_decode_inputs(w, seed=0)
    rates, desc, cores = [], "", 0
    for _ in range(args.warmup + args.steps):
        r, desc, cores, el = oracle_decode_sample(w, x, budget_s=0.0)   # one batch row per step
        rates.append(r)
    value = statistics.mean(rates[args.warmup:]) / 1e9
    line = {
        "impl": "reference", "metric": DECODE_METRIC, "value": value, "unit": DECODE_UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": decode_config(w, 1, "n/a (CPU)"),
        "cpu_baseline": {"value": value, "unit": DECODE_UNIT, "cores": cores, "kind": "oracle",
                         "sample": "each step: " + desc},
        "e2e": {"value": value, "unit": DECODE_UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- main
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_step: float, steps: int, max_ms: float) -> float:
    """Whole-job throughput: every rank runs the same per-step work (weak
    scaling), the job takes as long as its slowest rank."""
    return world * flops_per_step * steps / (max_ms / 1e3) / 1e12


def run_reference(args, world, rank):
    if rank != 0:
        return
    w = W.WORKLOADS[args.workload]
    x = W.make_inputs(w, seed=0)
    rates, descs, secs = [], [], 0.0
    cores = len(os.sched_getaffinity(0))
    for _ in range(args.warmup + args.steps):
        # one group per step, cut to a 1024-position causal prefix so that a
        # run of many steps stays within minutes
        r, d, cores, el = oracle_sample(w, x, budget_s=0.0, t_prefix=1024)
        rates.append(r)
        descs.append(d)
        secs += el
    timed = rates[args.warmup:]
    value = statistics.mean(timed) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "T": w.T, "D": w.D, "causal": w.causal,
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "each step: " + descs[-1]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=W.HEADLINE, choices=sorted(W.WORKLOADS) + sorted(W.DECODE_WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-parity", action="store_true", help="skip the oracle comparison before the timed steps")
    ap.add_argument("--no-graph", action="store_true", help="time eager calls, not replays of the step captured in a CUDA graph")
    ap.add_argument("--flush", default="read", choices=["read", "write", "none"],
                    help="L2 eviction between timed steps (see L2Flush)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup()
    if args.workload in W.DECODE_WORKLOADS:
        if args.impl == "reference":
            run_decode_reference(args, world, rank)
        else:
            run_decode(args, world, rank, local)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import causal_gqa_attention_fwd_gb300 as gq
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.WORKLOADS[args.workload]
    x = W.make_inputs(w, seed=rank)
    stream = torch.cuda.current_stream()
    varlen = w.varlen
    cu = x.get("cu_seqlens")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    scale = w.softmax_scale
    if varlen:
        cud = cu.to(dev)
        maxlen = x["max_seqlen"]
        o, lse = gq.attn_varlen_fwd(q, k, v, cud, maxlen, scale=scale)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(gq.attn_varlen_bwd_workspace_size(len(cu) - 1, q.shape[0], w.Hq, w.Hkv, w.D) + 256,
                         dtype=torch.uint8, device=dev)
    else:
        o, lse = gq.attn_fwd(q, k, v, scale=scale)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(gq.attn_bwd_workspace_size(w.B, w.Hq, w.Hkv, w.T, w.D), dtype=torch.uint8, device=dev)

    def step():
        if varlen:
            gq.attn_varlen_fwd(q, k, v, cud, maxlen, scale=scale, o=o, lse=lse)
            gq.attn_varlen_bwd(q, k, v, o, lse, do, cud, maxlen, scale=scale, dq=dq, dk=dk, dv=dv, workspace=ws)
        else:
            gq.attn_fwd(q, k, v, scale=scale, o=o, lse=lse)
            gq.attn_bwd(q, k, v, o, lse, do, scale=scale, dq=dq, dk=dk, dv=dv, workspace=ws)

    step()
    torch.cuda.synchronize()
    # The timed steps replay the step captured in a CUDA graph (the calls
    # allocate nothing and never synchronise), so that host-side launch
    # work does not set the pace of the small workloads; --no-graph times
    # the eager calls instead.
    graph = None
    if not args.no_graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize()
    run = graph.replay if graph is not None else step

    flush = L2Flush(args.flush, dev)
    f_fwd, f_bwd = flops(w, cu)
    for _ in range(args.warmup):
        flush(1)
        run()
    torch.cuda.synchronize()
    assert gq.get_device_status() == 0, "device status after warm-up"

    parity = None
    if rank == 0 and not args.no_parity:
        parity = parity_leg(w, x, dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv))

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    clocks.mark(0)
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush(i)
        ev[i][0].record(stream)
        run()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t_wall
    clocks.mark(1)
    # per-kernel events in a second pass of as many steps, so the timed
    # steps above carry no event records between their kernels
    gq.profile_reset()
    gq.profile_enable(True)
    for i in range(args.steps):
        flush(i)
        step()
    torch.cuda.synchronize()
    gq.profile_enable(False)
    prof = gq.profile_read()
    clk = clocks.stop()
    status = gq.get_device_status()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    local_ms = sum(step_ms)
    total_ms = max_over_ranks(world, local_ms)
    ms_per_step = total_ms / args.steps
    value = whole_job_tflops(world, f_fwd + f_bwd, args.steps, total_ms)
    n_fwd, t_fwd = prof["attn_fwd"]
    n_main, t_main = prof["bwd_dkdv"]
    bwd_ms = sum(prof[k][1] for k in ("bwd_pre", "bwd_dkdv", "bwd_dq")) / args.steps
    fwd_ms = t_fwd / max(n_fwd, 1)
    pk = peaks()
    gpu_launches = sum(prof[k][0] for k in prof)

    # roofline of the dominant kernel, the key/value-stationary dK/dV kernel,
    # whose algorithmic work is its four products per visible (query, key)
    # pair (S^T, dP^T, dV, dK: 8*D FLOPs; the separate dQ kernel does the
    # fifth and recomputes S and dP).
    main_ms = t_main / max(n_main, 1)
    main_flops = f_bwd * 0.8
    achieved = main_flops / (main_ms / 1e3) / 1e12
    roofline_traffic = measured_traffic(w.name, "bwd_dkdv")
    roofline = {"kernel": "bwd_dkdv", "bound": "tensor", "achieved": achieved,
                "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                "traffic": roofline_traffic, "peak_source": pk["source"] + " (burst bf16)",
                "flops_per_launch": main_flops,
                "flops_per_launch_basis": "8*D per visible (query, key) pair: S^T, dP^T, dV, dK"}

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hdo = (t.pin_memory() for t in (x["q"], x["k"], x["v"], x["do"]))
        ho, hlse = torch.empty_like(hq).pin_memory(), torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        hdq, hdk, hdv = (torch.empty_like(t).pin_memory() for t in (hq, hk, hv))
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hdo)) + (cu.numel() * 4 if varlen else 0)
        d2h = sum(t.numel() * t.element_size() for t in (ho, hlse, hdq, hdk, hdv))

        def e2e_step():
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            do.copy_(hdo, non_blocking=True)
            if varlen:
                cud.copy_(cu, non_blocking=True)
            step()
            ho.copy_(o, non_blocking=True)
            hlse.copy_(lse, non_blocking=True)
            hdq.copy_(dq, non_blocking=True)
            hdk.copy_(dk, non_blocking=True)
            hdv.copy_(dv, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        n_e2e = max(3, min(args.steps, 20))
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        torch.cuda.synchronize()
        serial_s = max_over_ranks(world, time.perf_counter() - t0)

        # The same steps double-buffered, as a training or serving loop runs
        # them: two sets of device buffers; step i's inputs cross on a copy-in
        # stream and step i's results on a copy-out stream, so they overlap
        # the kernels of steps i - 1 and i + 1.  Every step still moves all of
        # its h2d and d2h bytes inside the timed region.
        sets = []
        for _ in range(2):
            d = {n: torch.empty_like(t) for n, t in (("q", q), ("k", k), ("v", v), ("do", do), ("o", o),
                                                     ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv), ("ws", ws))}
            if varlen:
                d["cu"] = torch.empty_like(cud)
            hout = {n: torch.empty_like(t).pin_memory() for n, t in (("o", ho), ("lse", hlse), ("dq", hdq),
                                                                       ("dk", hdk), ("dv", hdv))}
            sets.append((d, hout))
        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        ev_in, ev_cmp, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
        used = [False, False]

        def piped_step(i):
            bset = i & 1
            d, hout = sets[bset]
            with torch.cuda.stream(s_in):
                if used[bset]:
                    s_in.wait_event(ev_cmp[bset])      # step i - 2 has finished reading these inputs
                for n, hsrc in (("q", hq), ("k", hk), ("v", hv), ("do", hdo)):
                    d[n].copy_(hsrc, non_blocking=True)
                if varlen:
                    d["cu"].copy_(cu, non_blocking=True)
                ev_in[bset].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[bset])
                if used[bset]:
                    s_cmp.wait_event(ev_out[bset])     # step i - 2's results have left these buffers
                if varlen:
                    gq.attn_varlen_fwd(d["q"], d["k"], d["v"], d["cu"], maxlen, scale=scale, o=d["o"], lse=d["lse"])
                    gq.attn_varlen_bwd(d["q"], d["k"], d["v"], d["o"], d["lse"], d["do"], d["cu"], maxlen,
                                       scale=scale, dq=d["dq"], dk=d["dk"], dv=d["dv"], workspace=d["ws"])
                else:
                    gq.attn_fwd(d["q"], d["k"], d["v"], scale=scale, o=d["o"], lse=d["lse"])
                    gq.attn_bwd(d["q"], d["k"], d["v"], d["o"], d["lse"], d["do"], scale=scale, dq=d["dq"],
                                dk=d["dk"], dv=d["dv"], workspace=d["ws"])
                ev_cmp[bset].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[bset])
                for n in ("o", "lse", "dq", "dk", "dv"):
                    hout[n].copy_(d[n], non_blocking=True)
                ev_out[bset].record(s_out)
            used[bset] = True

        for i in range(2):
            piped_step(i)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(n_e2e):
            piped_step(i)
        torch.cuda.synchronize()
        e2e_s = max_over_ranks(world, time.perf_counter() - t0)
        e2e = {"value": world * (f_fwd + f_bwd) * n_e2e / e2e_s / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "schedule": "double-buffered: copy-in, kernels and copy-out of successive steps on three streams",
               "serial_value": world * (f_fwd + f_bwd) * n_e2e / serial_s / 1e12,
               "serial_schedule": "each step's copies and kernels one after another on one stream"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, desc, cores, el = oracle_sample(w, x, args.cpu_budget)
        cpu = {"value": rate / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "T": w.T, "D": w.D,
                       "causal": w.causal, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": flush.describe(),
                       "launch": "CUDA graph replay of the step" if graph is not None else "eager calls"},
            "frac_of_peak": value / pk["bf16_tflops"],
            "fwd_tflops": f_fwd / (fwd_ms / 1e3) / 1e12,
            "bwd_tflops": f_bwd / (bwd_ms / 1e3) / 1e12,
            "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
            "kernel_ms": {k: (t / n if n else None) for k, (n, t) in prof.items()},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": gpu_launches,
            "kernel_ms_pass": "second pass, same steps, events per kernel (launches counted there)",
            "parity": parity,
            "clocks": clk,
            "device_status": status,
            "wall_s_timed_region": wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
