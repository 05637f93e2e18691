"""Benchmark of quantized-KV attention on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole hot path over one batch of synthetic input.
The default workload is the 16-layer decode step: 2 sequences x 200704
cached keys, 32 query / 4 KV heads, each layer's K and V codec drawn from
the f16 / q8_0 / q4_0 ladder; a step is the decode attention call of every
layer (other workloads add the append of the step's new tokens, a prefill
chunk, a re-encode or an eviction step).  Caches are built (untimed) through
the library's append kernel.  Inputs are resident in HBM when the timed
region starts; L2 is flushed (2 x L2 written, then read) before every timed
step.  Timing: CUDA events on the launching stream around each step, W
warm-up steps, K timed steps, barrier + synchronize on both sides, max over
ranks.  ``value`` is the whole-job effective bandwidth: algorithmic bytes
(every attended K/V row read once, q read, out written, appended rows read
and written) divided by the step time; ``us_per_layer_step`` is the step
time over the layers, and ``per_layer`` the time of each layer's call in a
replay of its own, with the mean per (K codec, V codec) pair.

Also reported: ``e2e`` (the same metric through the C ABI with pinned host
buffers: per step the H2D copy of q (and new K/V rows), the kernels, and the
D2H copy of the output), ``roofline`` for the dominant kernel, the SM clock
record of the timed region, and ``cpu_baseline``: the fp64 C oracle timed on
this host's cores on a bounded sample of the same workload, on all cores and
on one thread.

``--impl reference`` times that oracle alone (the reference arm) on the same
workload, metric and unit, without building or loading the CUDA library.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized-KV attention: effective HBM GB/s, % of peak, µs per layer-step"
DEFAULT_WORKLOAD = "decode_16layer_ladder_2x200704"
ROW = {0: 256, 1: 136, 2: 72, 3: 66}
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# ------------------------------------------------------------------ algorithmic work

def evict_work(w, lens, n_ev, ck, cv):
    """Algorithmic bytes of one probe-scored eviction step over sequences of
    the given lengths: (decode, probe, select, compact).  Decode reads K and V
    once; the probe reads K once more and reads and writes each token's score;
    the selection reads the middle scores and writes the list; compaction
    reads and writes the kept rows of both sides and their scores, and reads
    the list."""
    e = w.extra
    dec = sum(lens) * w.n_kv * (ROW[ck] + ROW[cv]) + len(lens) * w.n_q * (2 * 256 + 4)
    probe = sum(lens) * (w.n_kv * ROW[ck] + 8) + len(lens) * w.n_q * (256 + 4)
    mid = sum(max(0, n - e["n_sink"] - e["n_recent"]) for n in lens)
    sel = 4 * mid + 4 * sum(n_ev)
    kept = [n - k for n, k in zip(lens, n_ev)]
    comp = sum(kept) * (2 * w.n_kv * (ROW[ck] + ROW[cv]) + 8) + 4 * sum(n_ev)
    return dec, probe, sel, comp


def fused_decode_step(w) -> bool:
    """A decode step that appends one token per sequence runs as one fused
    call (attn_decode_append) per layer."""
    return w.kind == "decode" and w.append_new == 1


def step_work(w, fused=None):
    """(bytes, flops, roofline-kernel bytes per layer) of one step of workload
    w; the roofline kernel is the attention call (with the append's bytes when
    the step is fused), the re-encode, or (eviction steps) the compaction."""
    fused = fused_decode_step(w) if fused is None else fused
    lens = w.final_lens()
    total_b, total_f, per_layer = 0, 0, []
    for ck, cv in w.codecs:
        app = w.n_seqs * w.append_new * w.n_kv * (2 * 256 + ROW[ck] + ROW[cv])
        if w.kind == "evict":
            dec, probe, sel, comp = evict_work(w, lens, _workloads().n_evicted(w), ck, cv)
            per_layer.append(comp)
            total_b += dec + probe + sel + comp + app
            total_f += sum(lens) * w.n_q * 4 * 128 + sum(lens) * w.n_q * 2 * 128
            continue
        if w.kind == "degrade":
            src = ck if w.extra["side"] == 0 else cv
            kv = sum(lens) * w.n_kv * (ROW[src] + ROW[w.extra["dst"]])
            qo, fl = 0, 0
        elif w.kind == "decode":
            kv = sum(lens) * w.n_kv * (ROW[ck] + ROW[cv])
            qo = 2 * w.n_seqs * w.n_q * 256
            fl = sum(lens) * w.n_q * 4 * 128
        else:
            n_tok, q0 = w.append_new, w.lens[0]
            kv = (q0 + n_tok) * w.n_kv * (ROW[ck] + ROW[cv])
            qo = 2 * n_tok * w.n_q * 256
            fl = sum(q0 + i + 1 for i in range(n_tok)) * w.n_q * 4 * 128
        per_layer.append(kv + qo + (app if fused else 0))
        total_b += kv + qo + app
        total_f += fl
    return total_b, total_f, per_layer


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"kvq_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def wait_first(self, timeout=5.0):
        """Block until nvidia-smi has written its first sample (it takes a
        moment to start), so that the load window that follows is sampled."""
        t_end = time.perf_counter() + timeout
        while self.proc is not None and time.perf_counter() < t_end:
            self.f.flush()
            if os.path.getsize(self.path) > 0:
                return
            time.sleep(0.05)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ our arm

class OursArm:
    def __init__(self, w, device, fused=None):
        import torch
        import attention_quantized_kv_gb300 as kvq
        from attention_quantized_kv_gb300 import workloads as wl
        self.torch, self.kvq, self.wl, self.w, self.dev = torch, kvq, wl, w, device
        self.scale = 1.0 / math.sqrt(128)
        self.fused = fused_decode_step(w) if fused is None else fused
        self.layers, self.ws, self.q, self.kn, self.vn = [], [], [], [], []
        self.max_len = max(w.final_lens())
        self.init_lens = torch.tensor(w.lens, dtype=torch.int32, device=device)
        self.final_lens = torch.tensor(w.final_lens(), dtype=torch.int32, device=device)
        n_tok = w.append_new if w.kind == "prefill" else 1
        paged = bool(w.extra.get("paged"))
        if paged:
            table, n_pages = wl.page_table(w)
            table = torch.from_numpy(table).to(device)
        for l, (ck, cv) in enumerate(w.codecs):
            if paged:
                L = kvq.KVLayer(w.n_seqs, w.n_kv, w.n_q, w.capacity, ck, cv, device=device,
                                n_pages=n_pages, block_table=table)
            else:
                L = kvq.KVLayer(w.n_seqs, w.n_kv, w.n_q, w.capacity, ck, cv, device=device)
            self._fill(L, l)
            self.layers.append(L)
            qq = wl.queries(w, l, n_tok, device)
            if w.kind == "degrade":
                # the step's output: the re-encoded side, in its own buffer
                self.q.append(qq[:0, 0].contiguous())
                nb = kvq.kvq_cache_bytes(w.extra["dst"], w.n_seqs, w.n_kv, w.capacity)
            elif w.kind in ("decode", "evict"):
                self.q.append(qq[:, 0].contiguous())
                nb = kvq.attn_decode_workspace(L, self.max_len)
            else:
                self.q.append(qq[0].contiguous())
                nb = kvq.attn_prefill_workspace(L, w.lens[0], w.append_new)
            self.ws.append(torch.zeros(nb, dtype=torch.uint8, device=device))
            if w.append_new:
                ks = torch.stack([wl.kv_rows(w, l, 0, s, w.lens[s], w.append_new, device)
                                  for s in range(w.n_seqs)])
                vs = torch.stack([wl.kv_rows(w, l, 1, s, w.lens[s], w.append_new, device)
                                  for s in range(w.n_seqs)])
                self.kn.append(ks.contiguous())
                self.vn.append(vs.contiguous())
        self.n_new = torch.full((w.n_seqs,), w.append_new, dtype=torch.int32, device=device)
        self.out = [torch.empty_like(q) for q in self.q]
        self.lse = [torch.empty(q.shape[:2], dtype=torch.float32, device=device) for q in self.q]
        if w.kind == "evict":
            # running scores (reset to the probe history before every step),
            # the eviction lists and the compaction's second buffers
            e = w.extra
            self.scores0 = [wl.initial_scores(w, device) for _ in self.layers]
            self.scores = [s0.clone() for s0 in self.scores0]
            self.ev = [torch.zeros((w.n_seqs, e["n_evict"]), dtype=torch.int32, device=device)
                       for _ in self.layers]
            self.nev = [torch.zeros(w.n_seqs, dtype=torch.int32, device=device)
                        for _ in self.layers]
            self.k_dst = [torch.zeros_like(L.k_cache) for L in self.layers]
            self.v_dst = [torch.zeros_like(L.v_cache) for L in self.layers]
            self.s_dst = [torch.zeros_like(s0) for s0 in self.scores0]
            self.lens_dst = [torch.zeros(w.n_seqs, dtype=torch.int32, device=device)
                             for _ in self.layers]
        torch.cuda.synchronize()

    def _fill(self, L, l, chunk=8192):
        torch, wl, w = self.torch, self.wl, self.w
        for start in range(0, max(w.lens), chunk):
            n = [max(0, min(chunk, ln - start)) for ln in w.lens]
            mx = max(n)
            k = torch.zeros((w.n_seqs, mx, w.n_kv, 128), dtype=torch.float16, device=self.dev)
            v = torch.zeros_like(k)
            for s in range(w.n_seqs):
                if n[s]:
                    k[s, :n[s]] = wl.kv_rows(w, l, 0, s, start, n[s], self.dev)
                    v[s, :n[s]] = wl.kv_rows(w, l, 1, s, start, n[s], self.dev)
            self.kvq.kv_append_quantize(L, k, v, torch.tensor(n, dtype=torch.int32,
                                                              device=self.dev))

    def reset(self):
        for L in self.layers:
            L.seq_lens.copy_(self.init_lens)
        if self.w.kind == "evict":
            for sc, s0 in zip(self.scores, self.scores0):
                sc.copy_(s0)

    def set_final_lens(self):
        for L in self.layers:
            L.seq_lens.copy_(self.final_lens)

    def launches_per_step(self):
        """Kernels the library launches per step: the append is one kernel
        for at most 64 rows (it also advances the lengths), else the encode
        kernel plus the length update; decode is two (the split kernel, with
        the append fused when the step appends one token, and the merge),
        prefill three (dequant pre-pass, attention, merge of the split
        items), an eviction step five (decode's two, probe, selection,
        compaction of both sides)."""
        w = self.w
        per_layer = {"decode": 2, "degrade": 1, "prefill": 3, "evict": 5}[w.kind]
        if w.append_new and not self.fused:
            n_tok = w.append_new if w.kind == "prefill" else 1
            rows = 2 * w.n_seqs * n_tok * w.n_kv
            per_layer += 1 if rows <= 64 else 2
        return per_layer * len(self.layers)

    def step(self, q=None, kn=None, vn=None, out=None):
        """One pass of the hot path: every layer's append (when the workload
        has one) and attention call.  q / kn / vn / out: optional per-layer
        replacements of the resident tensors."""
        kvq, w = self.kvq, self.w
        for l, L in enumerate(self.layers):
            if self.fused:
                self.fused_step(l, q, kn, vn, out)
                continue
            if w.append_new:
                kvq.kv_append_quantize(L, (kn or self.kn)[l], (vn or self.vn)[l], self.n_new)
            self.attention(l, q, out)

    def fused_step(self, l, q=None, kn=None, vn=None, out=None):
        """One layer's decode step in one call: append the token, attend."""
        self.kvq.attn_decode_append(self.layers[l], (kn or self.kn)[l][:, 0],
                                    (vn or self.vn)[l][:, 0], (q or self.q)[l], self.scale,
                                    (out or self.out)[l], self.lse[l], self.max_len, self.ws[l])

    def roofline_calls(self, l):
        """The calls of the kernel the roofline line is about: the attention
        call, the re-encode, or (eviction steps) the compaction."""
        if self.w.kind == "evict":
            self.compact(l)
        elif self.fused:
            self.fused_step(l)
        else:
            self.attention(l)

    def compact(self, l):
        self.kvq.kv_compact(self.layers[l], self.ev[l], self.nev[l], self.k_dst[l],
                            self.v_dst[l], self.scores[l], self.s_dst[l], self.lens_dst[l])

    def attention(self, l, q=None, out=None):
        L, w = self.layers[l], self.w
        qq, oo = (q or self.q)[l], (out or self.out)[l]
        if w.kind == "evict":
            e = w.extra
            self.kvq.attn_decode(L, qq, self.scale, oo, self.lse[l], self.max_len, self.ws[l])
            self.kvq.kv_probe_scores(L, qq, self.scale, self.lse[l], e["decay"], self.scores[l])
            self.kvq.kv_evict_select(L, self.scores[l], e["n_sink"], e["n_recent"],
                                     e["n_evict"], self.ev[l], self.nev[l])
            self.compact(l)
        elif w.kind == "degrade":
            self.kvq.kv_requantize(L, w.extra["side"], w.extra["dst"], self.ws[l])
        elif w.kind == "decode":
            self.kvq.attn_decode(L, qq, self.scale, oo, self.lse[l], self.max_len, self.ws[l])
        else:
            self.kvq.attn_prefill_chunk(L, 0, w.lens[0], qq, self.scale, oo, self.lse[l],
                                        self.ws[l])

    def layer_errs(self):
        return [int(L.err.item()) for L in self.layers]


def _flush_l2(torch, bufs):
    """Evict the step's data from L2: write one scratch buffer larger than L2,
    then read another, so that L2 ends up holding clean unrelated lines (a
    flush by writes alone leaves ~L2-size dirty data whose write-back would be
    charged to the timed step).  bufs None (--warm): no flush."""
    if bufs is None:
        return
    wbuf, rbuf = bufs
    wbuf.zero_()
    rbuf.view(torch.int32).sum()


def _traffic_for(workload):
    """dram bytes per launch of the roofline kernel (decode, prefill attention
    or compaction) from a committed ncu summary, if it was taken on the
    current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("source_hash") != _kernel_source_hash(e.get("kernel", "decode")):
        return None
    return e.get("bytes_per_launch")


def _kernel_source_hash(kind):
    names = {"decode": ["decode.cu", "kvq_device.cuh", "kvq_encode.cuh"],
             "prefill": ["prefill.cu", "kvq_device.cuh"],
             "evict": ["evict.cu", "kvq_device.cuh"],
             "requant": ["append.cu", "kvq_device.cuh", "kvq_encode.cuh"]}[kind]
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "attention_quantized_kv_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def workload_config(w, world, l2, timing):
    """The line's config: the workload's shape (the same keys on both arms)
    plus how this arm was timed."""
    return {"workload": w.name, "description": w.description, "n_seqs": w.n_seqs,
            "n_q_heads": w.n_q, "n_kv_heads": w.n_kv, "head_dim": 128,
            "context": w.final_lens() if w.n_seqs <= 2 else
            {"sum": sum(w.final_lens()), "min": min(w.final_lens()), "max": max(w.final_lens())},
            "layers": w.n_layers,
            "codecs": [[["f16", "q8_0", "q4_0", "turbo4"][c] for c in p] for p in w.codecs],
            "l2": l2, "timing": timing, "parallelism": f"replicas x{world}"}


def reduce_max(dist, vals, device):
    """The per-rank timings reduced to their maximum over ranks (the job is as
    slow as its slowest replica); unchanged without a process group."""
    if not dist:
        return [float(v) for v in vals]
    import torch
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_gbps(world, bytes_step, steps, total_ms):
    """Whole-job throughput: every replica does bytes_step per step (weak
    scaling), over the slowest replica's time."""
    return world * bytes_step * steps / (total_ms * 1e-3) / 1e9


def run_ours(args, w, rank, world, dist):
    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    arm = OursArm(w, dev, fused=False if args.unfused else None)
    bytes_step, flops_step, per_layer_bytes = step_work(w, arm.fused)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)
    flush = None if args.warm else (torch.empty(2 * l2, dtype=torch.uint8, device=dev),
             torch.zeros(2 * l2, dtype=torch.uint8, device=dev))

    for _ in range(args.warmup):
        _flush_l2(torch, flush)
        arm.reset()
        arm.step()
    torch.cuda.synchronize()

    # The timed step is one CUDA graph replay of the whole step: every layer's
    # append and attention calls, captured through the C ABI, so that
    # consecutive kernels overlap through programmatic dependent launch.
    n_layers = len(arm.layers)
    arm.reset()
    g_step = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step):
        arm.step()
    # The attention calls alone, for the roofline of the attention kernels.
    # Timing events between the append and the attention kernel would cut
    # their overlap, so the attention calls are timed in a replay of their own
    # (lengths already final, L2 flushed the same way).
    g_attn = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_attn):
        for l in range(n_layers):
            arm.roofline_calls(l)
    # each layer's call alone (per-layer and per-codec-pair times)
    g_layer = []
    if n_layers > 1:
        for l in range(n_layers):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                arm.roofline_calls(l)
            g_layer.append(g)
    torch.cuda.synchronize()
    mode = ("one CUDA graph replay per step, events outside it; "
            + ("compaction kernels" if w.kind == "evict" else "attention kernels")
            + " timed in a replay of their own")
    if arm.fused:
        mode = ("one CUDA graph replay per step (one fused append + attention call per "
                "layer), events outside it")

    for _ in range(3):
        _flush_l2(torch, flush)
        arm.reset()
        g_step.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    # clocks: sampled over a ~1.5 s window of the same replayed steps that ends
    # with the timed region (the timed region alone is far shorter than one
    # nvidia-smi sample period)
    clk = ClockSampler(local)
    clk.start()
    clk.wait_first()
    t_end = time.perf_counter() + 1.5
    while time.perf_counter() < t_end:
        for _ in range(20):
            _flush_l2(torch, flush)
            arm.reset()
            g_step.replay()
        torch.cuda.synchronize()

    def timed(graph, prepare):
        ms = []
        for _ in range(args.steps):
            _flush_l2(torch, flush)
            prepare()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            graph.replay()
            b.record()
            b.synchronize()
            ms.append(a.elapsed_time(b))
        return ms

    step_ms = timed(g_step, arm.reset)
    attn_ms = timed(g_attn, arm.reset if arm.fused else arm.set_final_lens)
    layer_ms = [timed(g, arm.reset if arm.fused else arm.set_final_lens) for g in g_layer]
    torch.cuda.synchronize()
    clocks = clk.stop()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    total_ms = float(sum(step_ms))
    attn_bytes = sum(per_layer_bytes) * args.steps
    errs = arm.layer_errs()

    # e2e: through the C ABI with the step's inputs in one pinned host buffer
    # (one host-to-device copy) and its outputs gathered by one device-to-host
    # copy, both inside the timed region.  The copies and the calls are
    # captured together in one CUDA graph (a serving loop's decode step); if
    # this torch cannot capture the copies, they run eagerly.
    ins = arm.q + arm.kn + arm.vn
    n_in = sum(t.numel() for t in ins)
    h_in = torch.empty(n_in, dtype=torch.float16, pin_memory=True)
    d_in = torch.empty(n_in, dtype=torch.float16, device=dev)
    views, off = [], 0
    for t in ins:
        h_in[off:off + t.numel()].copy_(t.flatten().cpu())
        views.append(d_in[off:off + t.numel()].view(t.shape))
        off += t.numel()
    nl = len(arm.q)
    d_q, d_k, d_v = views[:nl], views[nl:nl + len(arm.kn)], views[nl + len(arm.kn):]
    n_out = sum(o.numel() for o in arm.out)
    d_out = torch.empty(n_out, dtype=torch.float16, device=dev)
    h_out = torch.empty(n_out, dtype=torch.float16, pin_memory=True)
    out_views, off = [], 0
    for o in arm.out:
        out_views.append(d_out[off:off + o.numel()].view(o.shape))
        off += o.numel()
    h2d = n_in * 2
    d2h = n_out * 2

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        arm.step(d_q, d_k or None, d_v or None, out_views)
        h_out.copy_(d_out, non_blocking=True)

    e2e_mode = "one CUDA graph per step: H2D copy, the calls, D2H copy"
    try:
        arm.reset()
        torch.cuda.synchronize()
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e):
            e2e_step()
        torch.cuda.synchronize()
        run_e2e = g_e2e.replay
    except Exception as exc:  # capture of pinned-host copies unsupported: eager
        torch.cuda.synchronize()
        run_e2e = e2e_step
        e2e_mode = f"eager calls (graph capture failed: {type(exc).__name__})"
    e2e_ms = []
    for it in range(args.warmup + args.steps):
        _flush_l2(torch, flush)
        arm.reset()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        run_e2e()
        b.record()
        b.synchronize()
        if it >= args.warmup:
            e2e_ms.append(a.elapsed_time(b))
    e2e_total = float(sum(e2e_ms))

    total_ms, e2e_total = reduce_max(dist, [total_ms, e2e_total], dev)
    if rank != 0:
        return None

    hbm, tf, peak_kind = _peaks()
    ms_step = total_ms / args.steps
    value = job_gbps(world, bytes_step, args.steps, total_ms)
    achieved_attn = attn_bytes / (sum(attn_ms) * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "us_per_layer_step": round(ms_step * 1e3 / n_layers, 3),
        "pct_of_hbm_peak": round(100 * value / world / hbm, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16 in / fp32 accumulate over q8_0/q4_0/f16 KV",
        "data": "synthetic (seeded N(0,1) fp16 draws, cache built by the append kernel)",
        "config": workload_config(
            w, world,
            l2=("not flushed: warm L2 (the step's data left there by the previous step)"
                if args.warm else
                "flushed before every timed step (2 x L2 write, then 2 x L2 read)"),
            timing=mode),
        "bytes_per_step": bytes_step,
        "flops_per_step": flops_step,
        "e2e": {"value": round(job_gbps(world, bytes_step, args.steps, e2e_total), 2),
                "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_total / args.steps, 5), "mode": e2e_mode},
        "gpu_launches": arm.launches_per_step() * args.steps,
        "clocks": clocks,
        "device_errors": errs,
    }
    if layer_ms:
        names = ["f16", "q8_0", "q4_0", "turbo4"]
        us = [float(np.mean(m)) * 1e3 for m in layer_ms]
        pairs = {}
        for l, (ck, cv) in enumerate(w.codecs):
            key = f"K {names[ck]} / V {names[cv]}"
            e = pairs.setdefault(key, {"layers": [], "us": [], "bytes": 0})
            e["layers"].append(l)
            e["us"].append(us[l])
            e["bytes"] += per_layer_bytes[l]
        line["per_layer"] = {
            "what": "each layer's call alone: one CUDA graph replay per timed step, L2 flushed",
            "us": [round(u, 2) for u in us],
            "by_codec_pair": {k: {"layers": e["layers"], "us_mean": round(float(np.mean(e["us"])), 2),
                                  "gbs": round(e["bytes"] / (sum(e["us"]) * 1e-6) / 1e9, 1),
                                  "frac_of_hbm": round(e["bytes"] / (sum(e["us"]) * 1e-6) / 1e9
                                                       / _peaks()[0], 4)}
                              for k, e in sorted(pairs.items())}}
    if w.kind in ("decode", "degrade", "evict"):
        kname = {"decode": "attn_decode_append (decode_split_kernel with the append fused, "
                           "decode_merge_kernel)" if arm.fused
                 else "attn_decode (decode_split_kernel, decode_merge_kernel)",
                 "degrade": "kv_requantize (rq_block_kernel; requant_kernel for turbo4)",
                 "evict": "kv_compact (compact_kernel)"}[w.kind]
        line["roofline"] = {"bound": "hbm", "kernel": kname,
                            "achieved": round(achieved_attn, 2), "peak": hbm,
                            "peak_kind": peak_kind, "unit": "GB/s",
                            "frac": round(achieved_attn / hbm, 4),
                            "traffic": _traffic_for(w.name)}
    else:
        tfs = flops_step / (np.mean(attn_ms) * 1e-3) / 1e12
        line["roofline"] = {"bound": "tensor", "kernel": "attn_prefill_chunk",
                            "achieved": round(tfs, 2), "peak": tf, "peak_kind": peak_kind,
                            "unit": "TFLOP/s", "frac": round(tfs / tf, 4),
                            "traffic": _traffic_for(w.name)}
    return line


# ------------------------------------------------------------------ the oracle (CPU)

class OracleArm:
    """The fp64 C oracle over a bounded sample of the workload on host cores.

    Decode samples whole (layer, seq, kv head) groups, in order, until the
    sample's attended (key, query head) pairs reach ``budget_rows``; one step
    is then one oracle decode call per sampled layer over all of that layer's
    sampled groups, so the oracle's threads spread over (group, query head)
    rows.  Prefill samples 4 query rows of every head."""

    def __init__(self, w, budget_rows=2e7):
        import torch
        import oracle
        wl = _workloads()
        self.w, self.oracle, self.scale = w, oracle, 1.0 / math.sqrt(128)
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        if w.kind == "evict":
            self._init_evict(wl, dev)
            return
        G = w.n_q // w.n_kv
        groups, budget = [], 0
        cap_rows = budget_rows if w.kind == "decode" else 0
        for l in range(w.n_layers):
            for s in range(w.n_seqs):
                for h in range(w.n_kv):
                    if groups and budget >= cap_rows:
                        break
                    groups.append((l, s, h))
                    budget += w.final_lens()[s] * G
        self.groups = groups
        # per sampled layer: the layer's caches (every group appended, the
        # unsampled ones are simply not attended), the new rows, the query
        self.layers = []
        for l in sorted({g[0] for g in groups}):
            sel = np.zeros((w.n_seqs, w.n_kv), bool)
            for (gl, s, h) in groups:
                if gl == l:
                    sel[s, h] = True
            seqs = [s for s in range(w.n_seqs) if sel[s].any()]
            ck, cv = w.codecs[l]
            cs = []
            for side, codec in ((0, ck), (1, cv)):
                c = np.zeros(oracle.cache_bytes(codec, w.n_seqs, w.n_kv, w.capacity), np.uint8)
                for s in seqs:
                    rows = wl.kv_rows(w, l, side, s, 0, w.lens[s], dev).cpu().numpy()
                    x = np.zeros((w.n_seqs, w.lens[s], w.n_kv, 128), np.float16)
                    x[s] = rows
                    n = [w.lens[s] if t == s else 0 for t in range(w.n_seqs)]
                    oracle.append_side(codec, side, c, w.n_seqs, w.n_kv, w.capacity,
                                       [0] * w.n_seqs, n, x)
                new = None
                if w.append_new:
                    new = np.stack([wl.kv_rows(w, l, side, s, w.lens[s], w.append_new, dev)
                                    .cpu().numpy() for s in range(w.n_seqs)])
                cs.append((c, new))
            n_tok = w.append_new if w.kind == "prefill" else 1
            qq = wl.queries(w, l, n_tok, dev).cpu().numpy()  # [n_seqs, n_tok, n_q, 128]
            self.layers.append((l, sel, cs, qq))
        self.rows = None
        if w.kind == "prefill":
            self.rows = [0, 1, w.append_new // 2, w.append_new - 1]
        self.sample_desc = (f"{len(groups)} of {w.n_layers * w.n_seqs * w.n_kv} "
                            f"(layer, seq, kv head) groups"
                            + (f", {len(self.rows)} of {w.append_new} query rows"
                               if self.rows else ""))

    def _init_evict(self, wl, dev):
        """Eviction steps need every kv head of a sequence (the probe sums over
        all query heads): the sample is whole sequences, in order, until the
        attended keys reach ~2e7 x query heads."""
        w, o = self.w, self.oracle
        (ck, cv), = w.codecs
        seqs, budget = [], 0
        for s in range(w.n_seqs):
            if seqs and budget > 1e6:
                break
            seqs.append(s)
            budget += w.final_lens()[s] * w.n_q
        self.seqs, self.ev_caches, self.ev_q, self.ev_sc = seqs, [], [], []
        sc0 = wl.initial_scores(w, dev).cpu().numpy()
        for s in seqs:
            n = w.lens[s]
            cs = []
            for side, codec in ((0, ck), (1, cv)):
                rows = wl.kv_rows(w, 0, side, s, 0, n, dev).cpu().numpy()
                c = np.zeros(o.cache_bytes(codec, 1, w.n_kv, w.capacity), np.uint8)
                o.append_side(codec, side, c, 1, w.n_kv, w.capacity, [0], [n],
                              rows.reshape(1, n, w.n_kv, 128))
                cs.append(c)
            self.ev_caches.append(cs)
            self.ev_q.append(wl.queries(w, 0, 1, dev)[s, 0].cpu().numpy())
            self.ev_sc.append(sc0[s])
        self.sample_desc = f"{len(seqs)} of {w.n_seqs} sequences (all kv heads)"
        self.groups = None

    def _step_evict(self):
        w, o, e = self.w, self.oracle, self.w.extra
        (ck, cv), = w.codecs
        for s, (kc, vc), q, sc in zip(self.seqs, self.ev_caches, self.ev_q, self.ev_sc):
            n = [w.final_lens()[s]]
            o.decode_layer(ck, cv, kc, vc, 1, w.n_kv, w.n_q, w.capacity, n, q[None], self.scale)
            mass = o.probe_mass(ck, kc, 1, w.n_kv, w.n_q, w.capacity, n, q[None], self.scale)
            score = (e["decay"] * sc.astype(np.float64) + mass[0]).astype(np.float32)
            ev = o.evict_select(score, n[0], e["n_sink"], e["n_recent"], e["n_evict"])
            o.compact_side(ck, 0, kc, 1, w.n_kv, w.capacity, n, [ev])
            o.compact_side(cv, 1, vc, 1, w.n_kv, w.capacity, n, [ev])

    def sample_bytes(self):
        w = self.w
        if w.kind == "evict":
            lens = [w.final_lens()[s] for s in self.seqs]
            n_ev = [_workloads().n_evicted(w)[s] for s in self.seqs]
            return sum(evict_work(w, lens, n_ev, *w.codecs[0]))
        tot = 0
        G = w.n_q // w.n_kv
        for (l, s, h) in self.groups:
            ck, cv = w.codecs[l]
            T = w.final_lens()[s]
            app = w.append_new * (2 * 256 + ROW[ck] + ROW[cv])
            if w.kind == "degrade":
                src = ck if w.extra["side"] == 0 else cv
                tot += T * (ROW[src] + ROW[w.extra["dst"]])
            elif w.kind == "decode":
                tot += T * (ROW[ck] + ROW[cv]) + 2 * G * 256 + app
            else:
                frac = len(self.rows) / w.append_new
                tot += frac * (T * (ROW[ck] + ROW[cv]) + 2 * w.append_new * G * 256) + app
        return tot

    def step(self):
        w, o = self.w, self.oracle
        if w.kind == "evict":
            self._step_evict()
            return
        for l, sel, cs, qq in self.layers:
            ck, cv = w.codecs[l]
            (kc, kn), (vc, vn) = cs
            if w.append_new:  # every step writes the same rows at the same positions
                n = [w.append_new] * w.n_seqs
                o.append_side(ck, 0, kc, w.n_seqs, w.n_kv, w.capacity, w.lens, n, kn)
                o.append_side(cv, 1, vc, w.n_seqs, w.n_kv, w.capacity, w.lens, n, vn)
            if w.kind == "degrade":
                side = w.extra["side"]
                o.requantize_side(ck if side == 0 else cv, w.extra["dst"], side,
                                  kc if side == 0 else vc, w.n_seqs, w.n_kv, w.capacity, w.lens)
            elif w.kind == "decode":
                o.decode_layer(ck, cv, kc, vc, w.n_seqs, w.n_kv, w.n_q, w.capacity,
                               w.final_lens(), np.ascontiguousarray(qq[:, 0]), self.scale,
                               sel=sel)
            else:
                o.prefill_chunk(ck, cv, kc, vc, w.n_kv, w.n_q, w.capacity, 0, w.lens[0],
                                np.ascontiguousarray(qq[0]), self.scale, rows=self.rows)


def _workloads():
    """The workload module, loaded from its file without importing the
    package (whose first use loads the CUDA library): the reference arm runs
    the oracle alone."""
    import importlib.util
    name = "kvq_bench_workloads"
    if name in sys.modules:
        return sys.modules[name]
    path = os.path.join(ROOT, "attention_quantized_kv_gb300", "workloads.py")
    spec = importlib.util.spec_from_file_location(name, path)
    mod = importlib.util.module_from_spec(spec)
    sys.modules[name] = mod
    spec.loader.exec_module(mod)
    return mod


def time_oracle(w, steps, warmup, min_seconds=0.0, threads=None, budget_rows=2e7):
    """Oracle throughput on a bounded sample: bytes of the sample per second,
    on `threads` OpenMP threads (None: all of the host's)."""
    import oracle
    arm = OracleArm(w, budget_rows)
    n_thr = oracle.num_threads() if threads is None else int(threads)
    with oracle.threads(n_thr):
        for _ in range(warmup):
            arm.step()
        t0 = time.perf_counter()
        n = 0
        while n < steps or (time.perf_counter() - t0) < min_seconds:
            arm.step()
            n += 1
            if min_seconds and n >= steps and time.perf_counter() - t0 >= min_seconds:
                break
        dt = time.perf_counter() - t0
    gbs = arm.sample_bytes() * n / dt / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": n_thr,
            "kind": "oracle", "sample": f"{arm.sample_desc}; {n} steps in {dt:.1f} s",
            "seconds": round(dt, 2)}


def cpu_baseline(w):
    """The oracle on all host cores (the reported value) and on one thread,
    each on its own bounded sample (~10 s each)."""
    import oracle
    allc = time_oracle(w, 1, 0, min_seconds=10.0, budget_rows=2e7)
    one = time_oracle(w, 1, 0, min_seconds=10.0, threads=1, budget_rows=2e6)
    allc["host_cores"] = os.cpu_count()
    allc["parallel_over"] = {
        "decode": "(kv head group, query head) rows of each sampled layer",
        "prefill": "query rows",
        "degrade": "tokens of each sampled stream",
        "evict": "decode: query rows; probe: tokens; compaction: (seq, kv head) streams; "
                 "selection: one thread",
    }[w.kind]
    allc["single_thread"] = {k: one[k] for k in ("value", "unit", "cores", "sample", "seconds")}
    return allc


# ------------------------------------------------------------------ main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--warm", action="store_true",
                    help="no L2 flush between steps (warm-cache numbers, reported as such)")
    ap.add_argument("--unfused", action="store_true",
                    help="one-token decode steps as two calls (append, then attention)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        if torch.cuda.is_available():
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        dist = tdist

    if args.impl == "reference":
        # the oracle alone: the CUDA library is neither built nor loaded here
        import oracle
        oracle.build()
        w = _workloads().get(args.workload)
        if rank == 0:
            r = time_oracle(w, args.steps, args.warmup, budget_rows=1e7)
            r["host_cores"] = os.cpu_count()
            line = {"metric": METRIC, "value": r["value"], "unit": "GB/s", "n_gpus": world,
                    "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
                    "scaling": "weak", "vs_baseline": None, "dtype": "f64 attention, fp32 codec",
                    "data": "synthetic", "impl": "reference",
                    "config": workload_config(
                        w, world, l2="not applicable (host CPU)",
                        timing="wall clock over whole oracle steps on a bounded sample"),
                    "cpu_baseline": r,
                    "e2e": {"value": r["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}
            print(json.dumps(line), flush=True)
        if dist:
            dist.destroy_process_group()
        return

    import __graft_entry__
    __graft_entry__.build()
    from attention_quantized_kv_gb300 import workloads as wl
    w = wl.get(args.workload)
    line = run_ours(args, w, rank, world, dist)
    if rank == 0:
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w)
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
