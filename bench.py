"""Decode-attention benchmark: µs per decode step and KV-read GB/s on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload long_ctx] [--impl gb300|reference]
                    [--l2 rotate|flush]

One step = one call of the whole path over the workload's batch: a single kernel launch that
computes the split-KV partials and, in the last CTA of each (row, KV head), their log-sum-exp
merge.  Prints ONE JSON line on rank 0.  Under torchrun (N > 1) every rank runs an
independent replica of the workload on its own GPU (weak scaling; the path needs no exchange).

Timing: W untimed warm-up steps, then K steps on the launching stream between CUDA events.
When the KV read of a step is at least 4x the 129 MB L2 (the default workload reads 941 MB),
the K steps run back to back between two events ("inputs larger than L2").  Smaller workloads
rotate: their cache-side inputs (K/V or packed cache, scales, ids, block scores) are copied n times
so that the copies hold at least 3x the L2, and the K steps run back to back between two events,
step i on copy i % n, so every step reads its cache from HBM.  By default the K steps are
captured into one CUDA graph (as a decode loop launches them) and timed as one replay, after an
untimed replay; ``--launch stream`` calls the library once per step from Python instead.
``--l2 flush`` times them one step at a time, with a 512 MiB device write before each step,
outside the step's events.
``value`` = algorithmic bytes per step (KV rows read once per KV head + q + out) / mean step time.
``e2e`` repeats the step through host buffers: pinned q and kv_len copied in, out copied back
every step.  For the large workloads it runs as a decode loop does, the copies on their own
stream with two device buffer sets so that they overlap the neighbouring steps' kernels (the
time is first upload to last download, over the steps); small workloads time one step at a
time, copies included.
``--impl reference`` times the fp64 CPU oracle on the host cores on a bounded sample per step.
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

# The CPU oracle legs run numpy with one BLAS thread per process (their core counts are the
# worker processes they fork); set before numpy loads its BLAS.  The GPU arm does no BLAS work.
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gqa_decode_attention_03_gb300 import workloads as W  # noqa: E402

METRIC = "decode-attention µs/step and KV-read GB/s (% of GB300 HBM peak), 1 GPU"
FLUSH_BYTES = 512 << 20
# GB300's nominal HBM3e bandwidth: the long-context batch's target (>= 70 % of HBM) is stated
# against about this figure; frac_of_hbm_peak is against the measured copy rate
# (MEASURED_PEAKS.json), which a pure read stream can exceed
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 << 20


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured bf16_tflops (MEASURED_PEAKS.json)"
    except Exception:
        return 1900.0, "fallback 1.9 PFLOP/s bf16"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _config(case, extra=None, l2_mode="rotate", copies=1, rot_bytes=0):
    big = case.kv_bytes() >= 4 * L2_BYTES
    small = ("flushed between steps: 512 MiB device write outside each step's events"
             if l2_mode == "flush" else
             f"rotated inputs: {copies} device copies of the step's cache-side inputs "
             f"({rot_bytes / 1e6:.0f} MB, >= 3x the 129 MB L2), steps back to back, each on "
             "the next copy")
    cfg = {"workload": case.name, "n_tok": int(case.n_tok), "n_heads": int(case.n_heads),
           "n_kv_heads": int(case.n_kv_heads), "head_dim": int(case.head_dim),
           "cache_cap": int(case.cache_cap), "kv_kind": case.kind,
           "visited_positions": int(sum(case.visited(t) for t in range(case.n_tok))),
           "seed": int(case.seed),
           "l2": (f"inputs larger than L2: {case.kv_bytes() / 1e6:.0f} MB of KV read per step vs "
                  "a 129 MB L2, steps back to back" if big else small)}
    if case.ids is not None:
        cfg["budget"] = int(case.budget)
    cfg.update(extra or {})
    return cfg


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, fl in rows for i, f in enumerate(fl)
                          if f.lower() == "active"})
        return {"sm_mhz": float(np.median([r[0] for r in rows])),
                "sm_max_mhz": float(max(r[1] for r in rows)), "reasons": reasons,
                "samples": len(rows)}


def _source_hash(sources=None):
    """Hash of the kernel sources a capture was taken on: the named files under csrc/ (all of
    them when none are named) and the public header."""
    import hashlib
    h = hashlib.sha1()
    csrc = os.path.join(ROOT, "gqa_decode_attention_03_gb300", "csrc")
    names = sorted(sources) if sources else sorted(
        n for n in os.listdir(csrc) if n.endswith((".cu", ".cuh", ".h")))
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    with open(os.path.join(ROOT, "include", "gqa_decode.h"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def _ncu_traffic(workload):
    """DRAM bytes per launch of the step's kernel from the committed ncu summary, when it was
    taken on the current sources of that kernel; otherwise None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        ent = d.get(workload)
        if ent and ent.get("source_hash") == _source_hash(ent.get("sources")):
            return float(ent["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def max_over_ranks(values):
    """Element-wise max of per-rank timings across the process group (the slowest rank sets the
    job's time); the identity without one.  Uses the group's own device: CUDA under NCCL, the
    CPU under gloo."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor(values, dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def _device_inputs(case, torch):
    d = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()  # noqa: E731
    if case.kind == "tq":
        w = lambda x: d(np.ascontiguousarray(x).view(np.int32))  # noqa: E731
        return {"q": d(case.q_rot), "q_jl": d(case.q_jl), "kv_len": d(case.kv_len),
                "seq_of": d(case.seq_of), "k_polar": w(case.k_polar), "k_jl": w(case.k_jl),
                "k_norms": w(case.k_norms), "v_polar": w(case.v_polar),
                "v_norms": w(case.v_norms), "signs": d(case.signs)}
    t = {"q": d(case.q), "kv_len": d(case.kv_len), "seq_of": d(case.seq_of)}
    if case.kind == "f16":
        t.update(k=d(case.k), v=d(case.v))
    else:
        t.update(kq=d(case.kq), vq=d(case.vq), ksc=d(case.ksc), vsc=d(case.vsc),
                 ids=None if case.ids is None else d(case.ids))
    return t


def _rows_fused_merge(plan, kind="f16"):
    """Grouped rows on the tcgen05 f16 kernel and on the TurboQuant row kernel merge their own
    partials when the grid fits one CTA per SM (the library's rule)."""
    if not (plan.merge and not plan.streamk and plan.row_group > 1):
        return False
    if kind != "tq" and os.environ.get("GQA_F16_ROWS") == "mma":
        return False
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return plan.grid_x * plan.grid_y * plan.grid_z <= sms


def _merge_launch(plan, kind="f16"):
    """1 when the step ends with a separate merge kernel (rows grouped by sequence)."""
    if (plan.merge and not plan.streamk and plan.row_group > 1
            and not _rows_fused_merge(plan, kind)):
        return 1
    return 0


def _precision(case, plan):
    """The operand precision of the step's contractions (all accumulate in fp32 and keep the
    online softmax in fp32; f16 K/V, int8 codes and TurboQuant bit planes enter exactly)."""
    if case.kind == "tq":
        return ("q_rot / q_jl and softmax weights as f16 hi + lo pairs (~22 bits); index and sign "
                "bit planes exact" + ("; centroids as f16 hi + lo planes" if plan.row_group > 1
                                      else "; centroids applied in fp32"))
    if plan.row_group > 1 and case.kind == "f16":
        if os.environ.get("GQA_F16_ROWS") == "mma":
            return "q and softmax weights as single f16 (11 bits) on mma.sync"
        return "q as f16 hi + lo (~22 bits); softmax weights as single f16 (11 bits) into P.V"
    return "q and softmax weights as f16 hi + lo pairs (~22 bits)"


def _kernel_name(case, plan):
    if case.kind == "tq":
        if plan.row_group > 1:
            if not plan.merge:
                return "tq_rows_kernel (rows grouped by sequence)"
            return "tq_rows_kernel (rows grouped by sequence" + (
                ", merge fused)" if _rows_fused_merge(plan, "tq") else ") + merge_kernel")
        name = "tq_decode_kernel" if os.environ.get("GQA_TQ_KERNEL") == "fma" else "tq_mma_kernel"
        return name + (" (split-KV, merge fused)" if plan.merge else "")
    if plan.streamk:
        return "streamk_mma_kernel (stream-K split, merge fused)"
    if plan.row_group > 1:
        rows = ("partial_mma_rows_kernel" if os.environ.get("GQA_F16_ROWS") == "mma"
                else "umma_rows_kernel")
        if not plan.merge:
            return rows + " (rows grouped by sequence)"
        if _rows_fused_merge(plan):
            return rows + " (rows grouped by sequence, merge fused)"
        return rows + " (rows grouped by sequence) + merge_kernel"
    if case.kind == "f16" and os.environ.get("GQA_F16_KERNEL") != "fma":
        name = "partial_mma_kernel"
    elif case.kind == "q8" and os.environ.get("GQA_Q8_KERNEL") != "fma":
        name = "partial_mma_q8_kernel"
    else:
        name = "partial_kernel"
    name += " (split-KV, merge fused)" if plan.merge else ""
    return ("select_cells_kernel + " + name) if "block_scores" in case.meta else name


def _e2e_pipelined(torch, step, stream, x, out, q_h, qj_h, kv_h, out_h, steps):
    """A decode loop through host buffers, as a server runs it: each step's inputs go up from
    pinned memory and its output comes back, on a copy stream with two device buffer sets, so
    that step i + 1's upload and step i's download overlap step i's and i + 1's kernels.
    Returns milliseconds per step over the whole loop (first upload to last download)."""
    copy = torch.cuda.Stream()
    nb = 2
    qd = [torch.empty_like(x["q"]) for _ in range(nb)]
    kvd = [torch.empty_like(x["kv_len"]) for _ in range(nb)]
    qjd = [torch.empty_like(x["q"]) if qj_h is not None else None for _ in range(nb)]
    od = [torch.empty_like(out) for _ in range(nb)]
    up = [torch.cuda.Event() for _ in range(nb)]
    comp = [torch.cuda.Event() for _ in range(nb)]
    down = [torch.cuda.Event() for _ in range(nb)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def upload(i):
        j = i % nb
        with torch.cuda.stream(copy):
            if i >= nb:
                copy.wait_event(comp[j])  # step i - nb has read this buffer set
            qd[j].copy_(q_h, non_blocking=True)
            if qjd[j] is not None:
                qjd[j].copy_(qj_h, non_blocking=True)
            kvd[j].copy_(kv_h, non_blocking=True)
            up[j].record(copy)

    torch.cuda.synchronize()
    t0.record(copy)
    upload(0)
    for i in range(steps):
        j = i % nb
        if i + 1 < steps:
            upload(i + 1)
        stream.wait_event(up[j])
        if i >= nb:
            stream.wait_event(down[j])  # step i - nb's output has left this buffer
        step(qd[j], kvd[j], qjd[j], od[j])
        comp[j].record(stream)
        with torch.cuda.stream(copy):
            copy.wait_event(comp[j])
            out_h.copy_(od[j], non_blocking=True)
            down[j].record(copy)
    t1.record(copy)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps


# inputs a step reads from HBM (rotated for the small workloads); q, kv_len, seq_of stay put
_ROTATED = ("k", "v", "kq", "vq", "ksc", "vsc", "ids", "k_polar", "k_jl", "k_norms", "v_polar",
            "v_norms", "scores")


def _rotation(x, torch):
    """Copies of the step's large inputs whose total is at least 3x the L2 (cold-L2 timing of
    workloads smaller than the cache): step i reads copy i % n, so by the time a copy comes
    round again the n - 1 others have passed through the L2.  Returns one input dict per
    copy (views into stacked tensors)."""
    names = [k for k in _ROTATED if x.get(k) is not None]
    per_copy = sum(x[k].numel() * x[k].element_size() for k in names)
    n = max(2, min(8192, -(-3 * L2_BYTES // max(per_copy, 1))))
    stacked = {k: x[k].unsqueeze(0).repeat((n,) + (1,) * x[k].dim()) for k in names}
    return [dict(x, **{k: stacked[k][i] for k in names}) for i in range(n)]


def _capture(torch, step, seq):
    """One CUDA graph of len(seq) steps, step i on input dict seq[i], replayed once (untimed)
    so that the graph is uploaded and the caches and clocks are in their steady state."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step(x=seq[0], s=side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cs = torch.cuda.current_stream()
        for xi in seq:
            step(x=xi, s=cs)
    g.replay()
    torch.cuda.synchronize()
    return g


def run_gpu(args):
    import torch
    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    from gqa_decode_attention_03_gb300 import gqa_decode as gd

    case = W.NAMED[args.workload]()
    x = _device_inputs(case, torch)
    T, H, D, Hk = case.n_tok, case.n_heads, case.head_dim, case.n_kv_heads
    max_len = int(min(case.cache_cap, case.kv_len.max()))
    kind = {"f16": gd.KIND_F16, "q8": gd.KIND_Q8, "tq": gd.KIND_TQ}[case.kind]
    budget = -1 if case.ids is None else int(case.budget)
    plan = gd.plan(T, H, Hk, D, max_len, budget, kind, n_seq=case.n_seq)
    ws = gd.alloc_workspace(T, H, Hk, D, max_len, budget, kind, n_seq=case.n_seq)
    out = torch.empty((T, H, D), dtype=torch.float32, device="cuda")
    stream = launch = torch.cuda.current_stream()

    scores = case.meta.get("block_scores")
    if scores is not None:  # the step chooses its ids first (block top-k selection)
        x["scores"] = torch.from_numpy(scores).cuda()
        x["ids"] = torch.empty((T, case.budget), dtype=torch.int32, device="cuda")

    def step(q=None, kv=None, q_jl=None, o=None, x=x, s=None):
        stream = launch if s is None else s  # s: a graph's capture stream
        q = x["q"] if q is None else q
        kv = x["kv_len"] if kv is None else kv
        o = out if o is None else o
        if case.kind == "tq":
            gd.attn_decode_tq(q, x["q_jl"] if q_jl is None else q_jl, x["k_polar"], x["k_jl"],
                              x["k_norms"], x["v_polar"], x["v_norms"], case.centroids,
                              x["signs"], case.qjl_scale, kv, scale=case.scale,
                              seq_of=x["seq_of"], max_kv_len=max_len, out=o, ws=ws,
                              stream=stream)
            return
        if scores is not None:
            gd.attn_select_topk(x["scores"], kv, case.budget, max_kv_len=case.cache_cap,
                                ids=x["ids"], stream=stream)
        if case.kind == "f16":
            gd.attn_decode_f16(q, x["k"], x["v"], kv, scale=case.scale, seq_of=x["seq_of"],
                               max_kv_len=max_len, out=o, ws=ws, stream=stream)
        else:
            gd.attn_decode_q8_sel(q, x["kq"], x["vq"], x["ksc"], x["vsc"], kv, ids=x["ids"],
                                  budget=None if x["ids"] is None else case.budget,
                                  scale=case.scale, seq_of=x["seq_of"], max_kv_len=max_len,
                                  out=o, ws=ws, stream=stream)

    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    big = case.kv_bytes() >= 4 * L2_BYTES
    rot = _rotation(x, torch) if not big and args.l2 == "rotate" else [x]
    for i in range(args.warmup):
        flush.zero_()
        step(x=rot[i % len(rot)])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    K = args.steps
    graph = None
    if args.launch == "graph" and (big or args.l2 == "rotate"):
        graph = _capture(torch, step, [x] * K if big else [rot[i % len(rot)] for i in range(K)])
    with ClockSampler(local) as clk:
        if graph:
            # the K steps (each on its input copy, as below) replayed from one CUDA graph, the
            # launch path of a decode loop; a first replay, untimed, uploaded it
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            graph.replay()
            b.record()
            torch.cuda.synchronize()
            step_ms = np.array([a.elapsed_time(b) / K])
        elif big:
            # inputs far larger than L2: K back-to-back steps between two events
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(K):
                step()
            b.record(stream)
            torch.cuda.synchronize()
            step_ms = np.array([a.elapsed_time(b) / K])
        elif args.l2 == "flush":
            # small inputs: a 512 MiB device write between steps, outside each step's events
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(K)]
            for i in range(K):
                flush.zero_()
                ev[i][0].record(stream)
                step()
                ev[i][1].record(stream)
            torch.cuda.synchronize()
            step_ms = np.array([e0.elapsed_time(e1) for e0, e1 in ev])
        else:
            # small inputs: K back-to-back steps between two events, step i on input copy
            # i % n (n copies >= 3x the L2: every step reads its K/V from HBM)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(K):
                step(x=rot[i % len(rot)])
            b.record(stream)
            torch.cuda.synchronize()
            step_ms = np.array([a.elapsed_time(b) / K])
    if world > 1:
        torch.distributed.barrier()

    # end to end through host buffers: pinned q / kv_len in, out back, every step
    q_host = case.q_rot if case.kind == "tq" else case.q
    q_h = torch.from_numpy(q_host).pin_memory()
    qj_h = torch.from_numpy(case.q_jl).pin_memory() if case.kind == "tq" else None
    kv_h = torch.from_numpy(case.kv_len).pin_memory()
    out_h = torch.empty((T, H, D), dtype=torch.float32).pin_memory()
    Ke = min(K, 500)
    if big:
        e2e_ms = _e2e_pipelined(torch, step, stream, x, out, q_h, qj_h, kv_h, out_h, Ke)
    else:
        # small steps, L2 flushed before each: one step at a time, its copies in its events
        q_d, kv_d = torch.empty_like(x["q"]), torch.empty_like(x["kv_len"])
        qj_d = torch.empty_like(x["q"]) if qj_h is not None else None
        eve = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(Ke)]
        for a, b in eve:
            flush.zero_()
            a.record(stream)
            q_d.copy_(q_h, non_blocking=True)
            if qj_d is not None:
                qj_d.copy_(qj_h, non_blocking=True)
            kv_d.copy_(kv_h, non_blocking=True)
            step(q_d, kv_d, qj_d)
            out_h.copy_(out, non_blocking=True)
            b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = float(np.mean([a.elapsed_time(b) for a, b in eve]))

    ms, e2e_ms = max_over_ranks([float(step_ms.mean()), e2e_ms])
    if rank != 0:
        return
    alg = case.algorithmic_bytes()
    peak, peak_src = _peaks()
    # algorithmic bytes over the step time: on the default workload a step is one kernel (the
    # split-KV partial kernel with its merge fused); multi-kernel steps name every kernel
    achieved = alg / (ms * 1e-3) / 1e9
    traffic = _ncu_traffic(case.name)
    gbs = world * alg / (ms * 1e-3) / 1e9
    h2d = int(q_host.nbytes + case.kv_len.nbytes + (case.q_jl.nbytes if qj_h is not None else 0))
    data = ("synthetic: seeded N(0,1) q and f16 K/V, NaN past each sequence's length"
            if case.kind == "f16" else
            "synthetic: seeded N(0,1) q, uniform int8 K/V codes in [-127, 127] with uniform f16 "
            "scales in [0.005, 0.02]; NaN scales past each length; sorted random cell ids"
            if case.kind == "q8" else
            "synthetic: seeded N(0,1) rotated / JL queries, uniform random 2-bit indices and sign "
            "bits, f16 norms, Lloyd-Max 2-bit centroids; NaN norms past each length")
    # The roof of the step's dominant kernel.  Per-row decode reads each K/V byte once at a few
    # flops per byte: HBM.  Rows sharing a sequence turn the step into a dense contraction on the
    # tensor cores (f16: ~64 flop per K/V byte; TurboQuant: ~490 per packed byte): the lower of
    # the two measured roofs at that intensity (ridge = dense bf16 rate / HBM rate, ~290 flop
    # per byte; f16 has the nominal bf16 rate).  TurboQuant decode is reported against HBM too,
    # although it is bound by instruction issue (the integer work of unpacking 2-bit fields into
    # MMA fragments, profiles/tq_mma_kernel_tq_long_ctx.md): its HBM fraction is the headroom.
    hbm_src = (f"{peak_src} hbm_gbs (MEASURED_PEAKS.json)" if peak_src == "measured"
               else "fallback 6.8 TB/s")
    tflops = case.flops() / (ms * 1e-3) / 1e12
    tpk, tsrc = _tensor_peak()
    intensity = case.flops() / alg
    contraction = plan.row_group > 1
    if contraction and intensity * peak * 1e9 >= tpk * 1e12:
        roofline = {"bound": "tensor", "kernel": _kernel_name(case, plan),
                    "achieved": round(tflops, 2), "peak": tpk, "peak_source": tsrc,
                    "unit": "TFLOP/s", "frac": round(tflops / tpk, 4), "traffic": traffic,
                    "flop_per_byte": round(intensity, 1), "hbm_achieved_gbs": round(achieved, 1),
                    "hbm_frac": round(achieved / peak, 4)}
    else:
        roofline = {"bound": "hbm", "kernel": _kernel_name(case, plan),
                    "achieved": round(achieved, 1), "peak": peak, "peak_source": hbm_src,
                    "unit": "GB/s", "frac": round(achieved / peak, 4),
                    "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4), "traffic": traffic,
                    "flop_per_byte": round(intensity, 1), "achieved_tflops": round(tflops, 3),
                    "tensor_peak_tflops": tpk, "tensor_frac": round(tflops / tpk, 5)}
        if case.kind == "tq" and not contraction:
            roofline["limiter"] = ("instruction issue: integer ALU pipe unpacking 2-bit fields "
                                   "and sign bits into f16 MMA fragments (ncu summary in profiles/)")
    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s",
        "us_per_step": round(ms * 1e3, 3), "frac_of_hbm_peak": round(gbs / world / peak, 4),
        "frac_of_nominal_hbm": round(gbs / world / NOMINAL_HBM_GBS, 4),
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "precision": _precision(case, plan),
        "data": data,
        "config": _config(case, {"algorithmic_bytes_per_step": alg, "chunk": plan.chunk,
                                 "n_split": plan.n_split, "parallelism": f"replicas x{world}",
                                 "launch": ("the K steps replayed from one CUDA graph" if graph
                                            else "one library call per step from Python")},
                          l2_mode=args.l2, copies=len(rot),
                          rot_bytes=len(rot) * sum(v.numel() * v.element_size()
                                                   for k, v in rot[0].items() if k in _ROTATED
                                                   and v is not None)),
        "roofline": roofline,
        "e2e": {"value": round(world * alg / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "us_per_step": round(e2e_ms * 1e3, 3),
                "h2d_bytes_per_step": h2d,
                "timing": "pipelined loop: copies on a second stream, two buffer sets"
                if big else "one step at a time, copies inside its events",
                "d2h_bytes_per_step": int(T * H * D * 4)},
        "gpu_launches": int(K * (1 + (scores is not None) + _merge_launch(plan, case.kind))),
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload)
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- CPU oracle arms

_CHILD_ENV = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}


def _oracle_pair(case, t, g):
    """The oracle on one (row, KV head) of the case: the G query heads of KV head g."""
    import oracle
    G = case.n_heads // case.n_kv_heads
    s = int(case.seq_of[t])
    L = case.kv_len[t:t + 1]
    if case.kind == "tq":
        sl = (slice(s, s + 1), slice(g, g + 1))
        return oracle.decode_tq(case.q_rot[t:t + 1, g * G:(g + 1) * G],
                                case.q_jl[t:t + 1, g * G:(g + 1) * G], case.k_polar[sl],
                                case.k_jl[sl], case.k_norms[sl], case.v_polar[sl],
                                case.v_norms[sl], case.centroids, case.signs, case.qjl_scale,
                                case.scale, L, seq_of=[0])
    q = case.q[t:t + 1, g * G:(g + 1) * G]
    if case.kind == "f16":
        return oracle.decode_f16(q, case.k[s:s + 1, :, g:g + 1], case.v[s:s + 1, :, g:g + 1], L,
                                 case.scale, seq_of=[0])
    ids = None if case.ids is None else case.ids[t:t + 1]
    return oracle.decode_q8(q, case.kq[s:s + 1, :, g:g + 1], case.vq[s:s + 1, :, g:g + 1],
                            case.ksc[s:s + 1, :, g:g + 1], case.vsc[s:s + 1, :, g:g + 1], L,
                            case.scale, seq_of=[0], ids=ids, budget=case.budget)


def _pair_bytes(case, t):
    if case.kind == "tq":
        return case.visited(t) * case.pos_bytes()
    D = case.head_dim
    per_pos = 2 * D * 2 if case.kind == "f16" else 2 * (D + 2 * (D // case.scale_group))
    return case.visited(t) * per_pos


# The case a fork pool of oracle workers reads (set before the pool forks; copy-on-write).
_POOL_CASE = None


def _pool_pair(tg):
    t, g = tg
    _oracle_pair(_POOL_CASE, t, g)
    return _pair_bytes(_POOL_CASE, t)


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _run_pairs_parallel(case, pairs, cores):
    """The oracle over `pairs` on `cores` worker processes (forked from a process that holds no
    CUDA context); returns (seconds, KV bytes)."""
    import multiprocessing as mp
    global _POOL_CASE
    _POOL_CASE = case
    ctx = mp.get_context("fork")
    with ctx.Pool(cores) as pool:
        pool.map(_pool_pair, pairs[:cores], chunksize=1)  # workers up and warm
        t0 = time.perf_counter()
        nbytes = sum(pool.map(_pool_pair, pairs, chunksize=1))
        dt = time.perf_counter() - t0
    return dt, nbytes


def _baseline_child(workload, budget_s):
    """Runs in a child process with single-threaded BLAS: the oracle over the workload's
    (row, KV head) pairs on one core (until about budget_s / 3 seconds of work), then on every
    host core (one forked worker per core, the whole list of pairs repeated until about
    budget_s / 2 seconds); returns the all-core GB/s of KV processed, the one-core figure
    beside it."""
    case = W.NAMED[workload]()
    pairs = [(t, g) for t in range(case.n_tok) for g in range(case.n_kv_heads)]
    done, nbytes, t0 = 0, 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s / 3 and done < len(pairs):
        t, g = pairs[done]
        _oracle_pair(case, t, g)
        nbytes += _pair_bytes(case, t)
        done += 1
    dt1 = time.perf_counter() - t0
    one = {"value": round(nbytes / dt1 / 1e9, 4), "unit": "GB/s", "cores": 1,
           "sample": f"{done} of {len(pairs)} pairs, {nbytes / 1e6:.1f} MB of KV in {dt1:.1f} s"}
    cores = _cores()
    # repeat the pair list so the all-core run lasts about budget_s / 2 seconds
    per_pass = dt1 * len(pairs) / max(done, 1) / cores
    reps = max(1, min(4096, int(budget_s / 2 / max(per_pass, 1e-4))))
    dtn, nb = _run_pairs_parallel(case, pairs * reps, cores)
    return {"value": round(nb / dtn / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} x {len(pairs)} (row, KV head) pairs of {case.name}, "
                      f"{nb / 1e6:.1f} MB of KV in {dtn:.1f} s on {cores} forked workers, "
                      f"fp64 numpy, 1 BLAS thread each",
            "host_cores": os.cpu_count(), "single_core": one}


def cpu_baseline(workload, budget_s=20.0):
    env = dict(os.environ, **_CHILD_ENV)
    code = (f"import sys, json; sys.path.insert(0, {ROOT!r}); import bench; "
            f"print(json.dumps(bench._baseline_child({workload!r}, {budget_s})))")
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=600)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except Exception as e:  # the baseline is reported, never required
        return {"value": None, "unit": "GB/s", "cores": _cores(), "kind": "oracle",
                "sample": f"failed: {e!r}"[:200]}


def run_reference(args):
    """The fp64 CPU oracle as the reference arm, on every host core: each step is one batch of
    (row, KV head) pairs of the workload, one pair per core, run by a pool of forked worker
    processes (single-threaded numpy each), cycling through the pairs; rank 0 only."""
    import multiprocessing as mp
    global _POOL_CASE
    world, rank, _ = _dist()
    if rank != 0:
        return
    case = W.NAMED[args.workload]()
    pairs = [(t, g) for t in range(case.n_tok) for g in range(case.n_kv_heads)]
    cores = _cores()
    _POOL_CASE = case
    batch = lambda i: [pairs[(i * cores + j) % len(pairs)] for j in range(cores)]  # noqa: E731
    with mp.get_context("fork").Pool(cores) as pool:
        for i in range(args.warmup):
            pool.map(_pool_pair, batch(i), chunksize=1)
        nbytes, t0 = 0, time.perf_counter()
        for i in range(args.steps):
            nbytes += sum(pool.map(_pool_pair, batch(args.warmup + i), chunksize=1))
        dt = time.perf_counter() - t0
    gbs = nbytes / dt / 1e9
    sample = (f"{args.steps} steps, each {cores} (row, KV head) pairs of {case.name} (one per "
              f"core) cycling through {len(pairs)} pairs; fp64 numpy oracle, 1 BLAS thread per "
              f"worker process")
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (same seeded workload as the GPU arm)",
            "config": _config(case),
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="long_ctx", choices=sorted(W.NAMED))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--launch", default="graph", choices=["graph", "stream"],
                    help="timed steps replayed from one CUDA graph (default) or launched one "
                         "call at a time from Python (--l2 flush always launches per call)")
    ap.add_argument("--l2", default="rotate", choices=["rotate", "flush"],
                    help="cold L2 for workloads smaller than 4x the L2: rotate input copies "
                         "(steps back to back) or flush with a 512 MiB write before each step")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
