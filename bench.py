"""Benchmark of the layer-streamed decoder training step on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config 14b] [--impl reference]

Prints ONE JSON line (rank 0).  A step is one full call of the library's
training step: forward over every layer streamed from host tiles, LM head and
loss, backward with block recompute, gradient evacuation and Adam on every
host tile.  `value` is tokens/s with the tokens already in device memory;
`e2e` is the same step through the host-token C-ABI call with the tokens in
pinned host memory and the loss read back on the host.  Both include the
host<->device weight/gradient streaming, which is the method itself.

The default workload is the 14B-shaped GQA decoder (48 layers, d 5120, 40/8
heads x 128, ffn 13824, vocab 152064, batch 8 x seq 4096).  When the host
cannot hold all 48 layers' tiles the depth is truncated to what fits and the
JSON says so.  With `--impl reference` the CPU oracle is timed instead on a
bounded sample of the same workload (see `cpu_sample`).

N > 1 (torchrun): N data-parallel replicas of one model, one per GPU, each on
its own batch, whose gradients the runtime sums in host shared memory (one
copy of the host tiles; no collective on the data path); value = all ranks'
tokens / the slowest rank's time.  --independent-replicas runs N unrelated
models instead.
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

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import mt_inputs  # noqa: E402

METRIC = "streamed train tokens/s and MFU on 1 GB300; % of step roofline; H2D/D2H overlap"
# Workloads whose description fixes no checkpoint interval: their layers keep
# their internals in device memory where it holds them (no recompute).  The
# others follow their stated interval (every layer, every 2 layers).
KEEP_AUTO_WORKLOADS = ("14b", "70b")
NOMINAL_BF16_PFLOPS = 2.25


def _env_int(k, d):
    try:
        return int(os.environ.get(k, d))
    except ValueError:
        return d


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return j, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def gemm_traffic_per_flop():
    """DRAM bytes per GEMM FLOP of the GEMM kernel from the committed ncu
    summary of two full-shape 14B GEMM kinds (profiles/gemm_dram_14b_shapes.md),
    or None when gemm.cu has changed since the counters were taken (the
    summary records the source's SHA-256)."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", "gemm_dram_14b_shapes.md")
    src = os.path.join(ROOT, "host_memory_streamed_gb300", "csrc", "gemm.cu")
    if not (os.path.exists(prof) and os.path.exists(src)):
        return None
    fields = {}
    for line in open(prof):
        if ":" in line and line.startswith("- "):
            k, v = line[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if fields.get("gemm.cu sha256") != digest or "traffic bytes per GEMM flop" not in fields:
        return None
    return float(fields["traffic bytes per GEMM flop"])


def mem_available_bytes():
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def tile_bytes(s):
    """Host bytes of every tile kind (12 B/param + page padding), from the layout rules."""
    def sect(numels):
        off = 0
        for n in numels:
            off = (off + n * 2 + 255) // 256 * 256
        w = (off + 4095) // 4096 * 4096
        return 6 * w  # W + G (BF16) + M + V (FP32)
    q, kv = s.n_heads * s.head_dim, s.n_kv_heads * s.head_dim
    layer = sect([s.d_model, (q + 2 * kv) * s.d_model, s.d_model * q, s.d_model, 2 * s.ffn * s.d_model,
                  s.d_model * s.ffn])
    embed = sect([s.vocab * s.d_model])
    head = sect([s.d_model, s.vocab * s.d_model])
    return layer, embed, head


def fit_depth(s, n_replicas=1, margin=14 << 30):
    """Most layers whose host tiles fit in MemAvailable (per replica)."""
    avail = mem_available_bytes()
    layer, embed, head = tile_bytes(s)
    if avail is None:
        return s.n_layers
    per = (avail - margin) // max(1, n_replicas)
    L = int((per - embed - head) // layer)
    return max(1, min(s.n_layers, L))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), power=float(f[3]), hw=f[5], hwt=f[6], swt=f[7],
                                 swp=f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        reasons = set()
        for r in rows:
            for k, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                            ("swp", "sw_power_cap")):
                if r[k].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


def link_bandwidth(device, nbytes=1 << 30):
    """Pinned H2D and D2H GB/s, each measured while the other direction runs."""
    h1 = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h2 = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d1 = torch.empty(nbytes, dtype=torch.uint8, device=device)
    d2 = torch.empty(nbytes, dtype=torch.uint8, device=device)
    s1, s2 = torch.cuda.Stream(device), torch.cuda.Stream(device)
    best = (0.0, 0.0)
    for _ in range(3):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        torch.cuda.synchronize(device)
        with torch.cuda.stream(s1):
            e[0].record()
            d1.copy_(h1, non_blocking=True)
            e[1].record()
        with torch.cuda.stream(s2):
            e[2].record()
            h2.copy_(d2, non_blocking=True)
            e[3].record()
        torch.cuda.synchronize(device)
        h2d = nbytes / (e[0].elapsed_time(e[1]) * 1e-3) / 1e9
        d2h = nbytes / (e[2].elapsed_time(e[3]) * 1e-3) / 1e9
        best = (max(best[0], h2d), max(best[1], d2h))
    del h1, h2, d1, d2
    return best


def _union(iv):
    """Sorted, merged copy of a list of (start, end) intervals."""
    out = []
    for a, b in sorted(iv):
        if out and a <= out[-1][1]:
            out[-1][1] = max(out[-1][1], b)
        else:
            out.append([a, b])
    return out


def _measure(iv):
    return sum(b - a for a, b in iv)


def _intersect(u, w):
    """Total length of the intersection of two merged interval lists."""
    i = j = 0
    tot = 0.0
    while i < len(u) and j < len(w):
        a, b = max(u[i][0], w[j][0]), min(u[i][1], w[j][1])
        if b > a:
            tot += b - a
        if u[i][1] < w[j][1]:
            i += 1
        else:
            j += 1
    return tot


def timeline_overlap(tl):
    """Copy/compute overlap of one step from its device timeline.

    tl: (kind, visit, t0_ms, t1_ms) spans from mt_get_timeline -- each visit's
    compute-stream span and every chunk copy on the H2D and D2H streams, timed
    by CUDA events around each copy.  overlap = |(H2D u D2H) n compute| /
    |H2D u D2H| over the unions of the spans; each direction is also reported
    on its own."""
    from host_memory_streamed_gb300 import _lib
    comp = _union([(a, b) for k, _, a, b in tl if k == _lib.SPAN_COMPUTE])
    h2d = _union([(a, b) for k, _, a, b in tl if k == _lib.SPAN_H2D])
    d2h = _union([(a, b) for k, _, a, b in tl if k == _lib.SPAN_D2H])
    cp = _union(h2d + d2h)
    tc = _measure(cp)
    return {"method": "device timeline (CUDA events around every chunk copy and every visit's compute span); "
                      "|(H2D u D2H) n compute| / |H2D u D2H|",
            "h2d_chunks": sum(1 for k, *_ in tl if k == _lib.SPAN_H2D),
            "d2h_chunks": sum(1 for k, *_ in tl if k == _lib.SPAN_D2H),
            "copy_ms": tc, "compute_ms": _measure(comp),
            "overlap": _intersect(cp, comp) / tc if tc else None,
            "h2d_overlap": _intersect(h2d, comp) / _measure(h2d) if h2d else None,
            "d2h_overlap": _intersect(d2h, comp) / _measure(d2h) if d2h else None}


def host_bandwidth(nbytes=2 << 30):
    """Host memory GB/s (read + write) of a large torch CPU copy on all cores."""
    a = torch.ones(nbytes, dtype=torch.uint8)
    b = torch.zeros(nbytes, dtype=torch.uint8)
    best = 0.0
    for _ in range(3):
        t0 = time.perf_counter()
        b.copy_(a)
        best = max(best, 2 * nbytes / (time.perf_counter() - t0) / 1e9)
    del a, b
    return best


def load_synthetic_weights(model, s, device):
    """N(0, 0.02) BF16 weights drawn on the GPU from per-tile seeds (1000 + tile), gains 1."""
    for i in range(model.n_tiles):
        g = torch.Generator(device=device)
        g.manual_seed(1000 + i)
        info = model.infos[i]
        raw = torch.zeros(info["w_bytes"], dtype=torch.uint8, device=device)
        for name, meta in info["tensors"].items():
            n = meta["numel"]
            o = meta["offset"]
            if name in ("g1", "g2", "gf"):
                t = torch.ones(n, dtype=torch.bfloat16, device=device)
            else:
                t = (torch.randn(n, generator=g, device=device, dtype=torch.float32) * 0.02).to(torch.bfloat16)
            raw[o:o + 2 * n] = t.view(torch.uint8)
        model.load_tile(i, 0, raw.cpu())
        del raw


def token_batches(s, steps, device, rank=0):
    gen = torch.Generator(device=device)
    out = []
    for n in range(steps):
        gen.manual_seed(2000 + n + 1 + 100003 * rank)
        out.append(torch.randint(0, s.vocab, (s.batch, s.seq + 1), generator=gen, device=device, dtype=torch.int32))
    return out


def cpu_sample(s, repeats=1):
    """Time the oracle (FP32, all host cores) on one decoder layer of the workload.

    Sample: forward + backward of one full-width layer on one whole sequence
    (the workload's S, capped at 4096 tokens: the oracle materialises the
    S x S score matrix of every head), then FP32 Adam on that layer's
    parameters.  The layer's time at the workload's T = B * S is B sequences
    plus one Adam update; the whole-model time is that x (layers + the LM
    head's FLOPs in layer units), giving tokens/s for the full model.
    """
    import oracle
    from oracle import OracleConfig
    torch.set_num_threads(os.cpu_count() or 1)
    seq = min(s.seq, 4096)
    cfg = OracleConfig.from_shape(s)
    lw = {k: v.float() for k, v in mt_inputs.layer_weights(s, 0).items()}
    gen = torch.Generator().manual_seed(7)
    x = torch.randn(1, seq, s.d_model, generator=gen)
    dy = torch.randn(1, seq, s.d_model, generator=gen) * 1e-3
    cos, sin = oracle.rope_cos_sin(seq, s.head_dim, s.rope_theta, torch.float32)
    t_seq, t_adam = [], []
    for _ in range(repeats):
        t0 = time.perf_counter()
        y, c = oracle.layer_forward(x, lw, cfg, cos, sin)
        _, grads = oracle.layer_backward(dy, c, lw, cfg, cos, sin)
        t1 = time.perf_counter()
        for k, w in lw.items():
            z = torch.zeros_like(w)
            oracle.adam_update(w.to(torch.bfloat16), grads[k].to(torch.bfloat16), z, z, 1, cfg,
                               dtype=torch.float32)
        t2 = time.perf_counter()
        t_seq.append(t1 - t0)
        t_adam.append(t2 - t1)
    ts, ta = statistics.median(t_seq), statistics.median(t_adam)
    n_seq = s.batch * s.seq / seq
    t_layer = n_seq * ts + ta
    q, kv = s.n_heads * s.head_dim, s.n_kv_heads * s.head_dim
    lin = s.d_model * (q + 2 * kv) + q * s.d_model + 3 * s.d_model * s.ffn
    head_in_layers = (s.d_model * s.vocab) / lin
    t_model = t_layer * (s.n_layers + head_in_layers)
    cpu = ""
    try:
        import platform
        cpu = platform.machine()
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    cpu += ", " + line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    short = " (shorter than the workload's sequence: attention's share is understated)" if seq < s.seq else ""
    return {"value": s.batch * s.seq / t_model, "unit": "tokens/s", "cores": torch.get_num_threads(),
            "kind": "oracle",
            "sample": (f"oracle FP32 fwd+bwd of one {s.name} layer on 1x{seq} tokens ({ts:.2f} s){short} and "
                       f"FP32 Adam of its parameters ({ta:.2f} s); layer at T = {s.batch * s.seq} = "
                       f"{n_seq:g} x that sequence + one Adam ({t_layer:.1f} s), scaled to the full model as "
                       f"{s.n_layers} layers + {head_in_layers:.2f} layer-equivalents of LM head"),
            "cpu": cpu, "sample_seconds": ts + ta, "layer_seconds": t_layer}


def gemm_case(args, s):
    """One GEMM kind of the workload's step at its full shape, repeated: a small
    case (a few GB on the device) for DRAM-traffic counters of the GEMM kernel.
    gate_up: a = SwiGLU(n2 W_gu^T) with the gate/up pairs kept (M = T, N = 2 ffn,
    K = d); dw_gu: dW_gu = dGU^T n2, both operands MN-major (M = 2 ffn, N = d,
    K = T).  Prints one JSON line with the launch's FLOPs and algorithmic bytes."""
    from host_memory_streamed_gb300 import _lib, ops
    device = torch.device("cuda", 0)
    T, d, f = s.batch * s.seq, s.d_model, s.ffn
    g = torch.Generator(device=device).manual_seed(5)
    rnd = lambda *shape: (torch.randn(*shape, generator=g, device=device) * 0.02).to(torch.bfloat16)
    if args.gemm_case == "gate_up":
        A, B = rnd(T, d), rnd(2 * f, d)
        out = torch.empty(T, f, device=device, dtype=torch.bfloat16)
        gu = torch.empty(T, 2 * f, device=device, dtype=torch.bfloat16)
        run = lambda: ops.gemm(A, B, out, _lib.EPI_SWIGLU, out2=gu)
        M, N, K = T, 2 * f, d
        alg = 2 * (A.numel() + B.numel() + out.numel() + gu.numel())
    else:
        A, B = rnd(T, 2 * f), rnd(T, d)
        out = torch.empty(2 * f, d, device=device, dtype=torch.bfloat16)
        run = lambda: ops.gemm_layout(A, B, out, a_mn=True, b_mn=True)
        M, N, K = 2 * f, d, T
        alg = 2 * (A.numel() + B.numel() + out.numel())
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        run()
    e1.record()
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / args.steps
    print(json.dumps({"gemm_case": args.gemm_case, "workload": s.name, "M": M, "N": N, "K": K,
                      "flops_per_launch": 2.0 * M * N * K, "algorithmic_bytes_per_launch": alg,
                      "ms_per_launch": ms, "tflops": 2.0 * M * N * K / (ms * 1e-3) / 1e12}), flush=True)


def attention_case(args, s):
    """The attention kernels alone at the workload's batch, sequence and heads
    (q/k/v of standard deviation 1.4, the scale the decoder produces): forward,
    then backward (delta, dK/dV, dQ), CUDA events around each.  Prints one JSON
    line; FLOPs are the causal forward's (4 hd S(S+1)/2 per batch and head) and
    2.5x that for the backward, the usual convention."""
    from host_memory_streamed_gb300 import ops
    device = torch.device("cuda", 0)
    B, S, Hq, Hkv, hd = s.batch, s.seq, s.n_heads, s.n_kv_heads, s.head_dim
    T, ld = B * S, (Hq + 2 * Hkv) * hd
    g = torch.Generator(device=device).manual_seed(1)
    qkv = (torch.randn(T, ld, device=device, generator=g) * 1.4).to(torch.bfloat16)
    do = torch.randn(T, Hq * hd, device=device, generator=g).to(torch.bfloat16)
    o = torch.empty(T, Hq * hd, device=device, dtype=torch.bfloat16)
    lse = torch.empty(B * Hq * S, device=device)
    delta = torch.empty(B * Hq * S, device=device)
    dqkv = torch.empty(T, ld, device=device, dtype=torch.bfloat16)
    st = torch.zeros(1, device=device, dtype=torch.int32)
    for _ in range(args.warmup):
        ops.attention_fwd(qkv, B, S, Hq, Hkv, hd, o, lse, st)
        ops.attention_bwd(qkv, B, S, Hq, Hkv, hd, o, lse, do, delta, dqkv, status=st)
    torch.cuda.synchronize(device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    tf = tb = 0.0
    for _ in range(args.steps):
        ev[0].record()
        ops.attention_fwd(qkv, B, S, Hq, Hkv, hd, o, lse, st)
        ev[1].record()
        ops.attention_bwd(qkv, B, S, Hq, Hkv, hd, o, lse, do, delta, dqkv, status=st)
        ev[2].record()
        torch.cuda.synchronize(device)
        tf += ev[0].elapsed_time(ev[1])
        tb += ev[1].elapsed_time(ev[2])
    if int(st.item()) != 0:
        raise SystemExit(f"attention kernels reported status {int(st.item())}")
    tf, tb = tf / args.steps, tb / args.steps
    fl = 4.0 * B * Hq * hd * S * (S + 1) / 2
    print(json.dumps({"attention_case": s.name, "B": B, "S": S, "heads": f"{Hq}q/{Hkv}kv x {hd}",
                      "fwd_ms": tf, "bwd_ms": tb, "fwd_tflops": fl / (tf * 1e-3) / 1e12,
                      "bwd_tflops_model": 2.5 * fl / (tb * 1e-3) / 1e12}), flush=True)


def run_reference(args, s, rank):
    """The reference arm: the oracle timed on the host cores.  A step is one
    bounded sample (cpu_sample); ms_per_step is its measured wall time and
    value the whole-model tokens/s that sample gives."""
    if rank != 0:
        return
    for _ in range(args.warmup):
        cpu_sample(s)
    t0 = time.perf_counter()
    vals = [cpu_sample(s) for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    v = statistics.median(x["value"] for x in vals)
    t = statistics.median(x["layer_seconds"] for x in vals)
    line = {"metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * wall / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": s.name, "layers": s.n_layers, "batch": s.batch, "seq": s.seq},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": vals[0]["cores"], "kind": "oracle",
                             "sample": vals[0]["sample"], "cpu": vals[0]["cpu"]},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "model_ms_per_step_extrapolated": 1e3 * s.batch * s.seq / v,
            "layer_seconds": t}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="14b", choices=sorted(mt_inputs.PRESETS))
    ap.add_argument("--layers", type=int, default=0, help="override the depth (0 = preset, truncated to host RAM)")
    ap.add_argument("--mlp-chunk-rows", type=int, default=-1,
                    help="MLP row chunk (0 = whole step; default: chunk only when the device arena would not fit)")
    ap.add_argument("--keep-layers", default="preset",
                    help="layers whose internals stay on the device from forward to backward: a number, 'auto' "
                         "(as many as fit) or 'preset' (auto where the workload fixes no checkpoint interval, "
                         "else 0)")
    ap.add_argument("--sync-adam", action="store_true",
                    help="each step waits for all of its Adam updates (default: they finish during the next "
                         "step, each before its tile is uploaded; the timed regions wait for all of them)")
    ap.add_argument("--slab-grads", action="store_true",
                    help="gradients through the pinned slabs and the accumulator's copy (default: straight into "
                         "the page-locked G sections of the tiles)")
    ap.add_argument("--staged-weights", action="store_true",
                    help="weights through the packer's pinned staging chunks (default: each upload's DMA reads "
                         "the page-locked W section of the tile)")
    ap.add_argument("--adam-threads", type=int, default=0,
                    help="CPU Adam workers (0: the library's default, 3/4 of the hardware threads)")
    ap.add_argument("--share-device", action="store_true",
                    help="every rank on cuda:0: exercises the N > 1 path on one GPU (the ranks only meet on the "
                         "host); the throughput it prints is not an N-GPU figure")
    ap.add_argument("--independent-replicas", action="store_true",
                    help="N > 1: N unrelated models, one per GPU (default: one model, N data-parallel replicas "
                         "summing their gradients on the host)")
    ap.add_argument("--no-double-buffer", action="store_true",
                    help="ablation: one device weight buffer, so no upload overlaps compute")
    ap.add_argument("--gemm-case", choices=["gate_up", "dw_gu"], default=None,
                    help="run one GEMM kind of the step at full shape (a small case for DRAM counters) and exit")
    ap.add_argument("--attention-case", action="store_true",
                    help="run the attention kernels alone at the workload's shape and exit")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local = _env_int("LOCAL_RANK", 0)
    s = mt_inputs.PRESETS[args.config]
    full_layers = s.n_layers
    if args.layers:
        s = s.with_(n_layers=args.layers)
    if args.impl == "reference":
        run_reference(args, s, rank)
        return
    if args.gemm_case:
        gemm_case(args, s)
        return
    if args.attention_case:
        attention_case(args, s)
        return

    import host_memory_streamed_gb300 as hms
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    device = torch.device("cuda", 0 if args.share_device else local)
    torch.cuda.set_device(device)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist
    group = world > 1 and not args.independent_replicas
    L = fit_depth(s, n_replicas=1 if group else world) if not args.layers else s.n_layers
    s = s.with_(n_layers=L)

    peaks, peak_kind = measured_peaks()
    h2d_bw, d2h_bw = link_bandwidth(device)
    host_bw = host_bandwidth()

    chunk = args.mlp_chunk_rows
    if chunk < 0:
        free, _ = torch.cuda.mem_get_info(device)
        chunk = 0 if hms.StreamedDecoder.required_device_bytes(s) < 0.9 * free else 65536
    t_init = time.perf_counter()
    # replicas share the host's cores: split the Adam workers (3/4 of the cores, the library's
    # own default for one process) between them instead of oversubscribing
    adam_threads = max(2, (os.cpu_count() or 4) * 3 // 4 // world) if world > 1 else 0
    if group:  # the last replica runs every Adam update of the group
        adam_threads = 0 if rank == world - 1 else 2
    if args.adam_threads:
        adam_threads = args.adam_threads
    keep = args.keep_layers
    if keep == "preset":
        keep = "auto" if s.name in KEEP_AUTO_WORKLOADS else 0
    elif keep != "auto":
        keep = int(keep)
    if chunk:
        keep = 0  # a chunked MLP keeps no per-layer activations
    flags = hms.MT_TIME_KERNELS | (hms.MT_NO_DOUBLE_BUFFER if args.no_double_buffer else 0) | \
        (0 if args.sync_adam else hms.MT_ASYNC_ADAM) | (0 if args.slab_grads else hms.MT_DIRECT_GRADS) | \
        (0 if args.staged_weights else hms.MT_DIRECT_WEIGHTS)
    kw = {}
    if group:
        from host_memory_streamed_gb300 import replicas
        kw["replica_group"] = (replicas.shared_group_name("mt-bench"), rank, world)
    model = hms.StreamedDecoder.from_shape(s, flags=flags, device=device, mlp_chunk_rows=chunk,
                                           n_adam_threads=adam_threads, keep_layers=keep, **kw)
    if not group or rank == 0:  # a group's tiles are shared: one replica writes them
        load_synthetic_weights(model, s, device)
    model.barrier()
    init_s = time.perf_counter() - t_init
    toks = token_batches(s, args.warmup + args.steps, device, rank)
    host_toks = [t.cpu().pin_memory() for t in toks]
    s_comp = model.streams[0]

    for i in range(args.warmup):
        model.train_step(toks[i])
    # ---- timed region: device-resident tokens
    stats = []
    model.sync()  # no Adam work of the warm-up steps inside the timed region
    if pg:
        pg.barrier()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(device.index) as clk:
        e0.record(s_comp)
        losses = []
        for i in range(args.steps):
            losses.append(model.train_step(toks[args.warmup + i]))
            stats.append(model.stats())
        model.sync()  # every Adam update of the timed steps inside the timed region
        e1.record(s_comp)
        torch.cuda.synchronize(device)
    overlap_tl = timeline_overlap(model.timeline())  # the last timed step
    if pg:
        pg.barrier()
    elapsed = e0.elapsed_time(e1) / 1e3
    if pg:
        t = torch.tensor([elapsed], dtype=torch.float64)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        elapsed = float(t[0])
    tokens_per_step = s.batch * s.seq
    value = world * args.steps * tokens_per_step / elapsed

    free_b, total_b = torch.cuda.mem_get_info(device)
    dev_mem = {"arena_bytes": model.arena_bytes, "device_used_bytes": total_b - free_b,
               "torch_max_allocated_bytes": torch.cuda.max_memory_allocated(device)}
    # ---- e2e: host tokens through the C-ABI, loss read on the host
    torch.cuda.synchronize(device)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(s_comp)
    for i in range(args.steps):
        model.train_step(host_toks[args.warmup + i])
    model.sync()
    f1.record(s_comp)
    torch.cuda.synchronize(device)
    e2e_elapsed = f0.elapsed_time(f1) / 1e3
    if pg:
        t = torch.tensor([e2e_elapsed], dtype=torch.float64)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        e2e_elapsed = float(t[0])
    e2e = world * args.steps * tokens_per_step / e2e_elapsed
    model_keep = model.keep_layers
    n_params = sum(info["n_params"] for info in model.infos)
    model.close()
    del model

    st = stats[-1]
    ms_step = 1e3 * elapsed / args.steps
    gemm_ms = sum(x["gemm_ms"] for x in stats)
    gemm_flops = sum(x["gemm_flops"] for x in stats)
    gemm_launches = sum(x["gemm_launches"] for x in stats)
    kernels = sum(x["kernel_launches"] for x in stats)
    p_sust = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    p_burst = peaks["bf16_tflops"]
    achieved = gemm_flops / (gemm_ms * 1e-3) / 1e12 if gemm_ms else None
    flops_exec = st["flops_executed"]
    flops_model = st["flops_model"]
    t_flops = flops_exec / (p_sust * 1e12)
    t_h2d = st["h2d_bytes"] / (h2d_bw * 1e9)
    t_d2h = st["d2h_bytes"] / (d2h_bw * 1e9)
    step_roof = max(t_flops, t_h2d, t_d2h)
    lin_bytes = st["h2d_bytes"] + st["d2h_bytes"]
    copy_ms = sum(x["h2d_ms"] + x["d2h_ms"] for x in stats)
    stall_ms = sum(x["wait_weights_ms"] for x in stats)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": s.name, "layers": s.n_layers, "layers_preset": full_layers, "d_model": s.d_model,
                   "heads": f"{s.n_heads}q/{s.n_kv_heads}kv x {s.head_dim}", "ffn": s.ffn, "vocab": s.vocab,
                   "batch": s.batch, "seq": s.seq, "ckpt_every": s.ckpt_every,
                   "keep_layers": model_keep, "double_buffer": not args.no_double_buffer,
                   "adam": "sync" if args.sync_adam else "async (finished inside the timed region)",
                   "grads": "pinned slabs + accumulator copy" if args.slab_grads else "direct into page-locked G",
                   "weights": "packer copy into pinned staging + DMA" if args.staged_weights
                   else "DMA from page-locked W",
                   "parallelism": ("data-parallel replica group" if group else "independent replicas")
                   if world > 1 else "single-gpu",
                   "l2": "inputs larger than L2 (weights streamed per layer, activations > 129 MB)",
                   "mlp_chunk_rows": chunk or None,
                   "truncated": s.n_layers < full_layers,
                   "truncation_reason": ("host RAM: tiles of all layers do not fit" if s.n_layers < full_layers
                                         and not args.layers else None)},
        "mfu": flops_model / (ms_step * 1e-3) / (NOMINAL_BF16_PFLOPS * 1e15),
        "mfu_vs_measured_peak": flops_model / (ms_step * 1e-3) / (peaks["bf16_tflops"] * 1e12),
        "executed_tflops": flops_exec / (ms_step * 1e-3) / 1e12,
        "step_roofline": {"flops_executed": flops_exec, "flops_model": flops_model, "t_flops_ms": 1e3 * t_flops,
                          "h2d_bytes": st["h2d_bytes"], "d2h_bytes": st["d2h_bytes"],
                          "h2d_gbs_measured": h2d_bw, "d2h_gbs_measured": d2h_bw, "t_h2d_ms": 1e3 * t_h2d,
                          "t_d2h_ms": 1e3 * t_d2h, "bound": "tensor" if t_flops >= max(t_h2d, t_d2h) else "link",
                          "frac": step_roof / (ms_step * 1e-3),
                          "peak": p_sust, "peak_kind": f"bf16_tflops_sustained ({peak_kind})",
                          "frac_vs_burst_peak": max(flops_exec / (p_burst * 1e12), t_h2d, t_d2h) / (ms_step * 1e-3),
                          "peak_burst": p_burst},
        "overlap": {"copy_ms_per_step": copy_ms / args.steps, "compute_stall_on_weights_ms_per_step":
                    stall_ms / args.steps,
                    "hidden_frac": (1.0 - stall_ms / copy_ms) if copy_ms else None,
                    "method": "CUDA events: copy windows on the H2D/D2H streams vs compute-stream waits",
                    "timeline": overlap_tl},
        "roofline": {"bound": "tensor", "kernel": "gemm_bf16_tcgen05", "achieved": achieved, "peak": p_sust,
                     "unit": "TFLOP/s", "frac": (achieved / p_sust) if achieved else None,
                     "traffic": (gemm_traffic_per_flop() * gemm_flops / max(1, gemm_launches)
                                 if s.name == "14b" and gemm_traffic_per_flop() else None),
                     "traffic_basis": "DRAM bytes per FLOP of two full-shape 14B GEMM kinds (ncu, "
                                      "profiles/gemm_dram_14b_shapes.md) x this step's FLOPs per GEMM launch",
                     "peak_kind": f"bf16_tflops_sustained ({peak_kind}) -- timed inside a long step",
                     "launches": gemm_launches, "flops_per_launch": gemm_flops / max(1, gemm_launches),
                     "ms_per_launch": gemm_ms / max(1, gemm_launches)},
        "e2e": {"value": e2e, "unit": "tokens/s",
                "h2d_bytes_per_step": 4 * (3 * tokens_per_step + s.vocab + 1) + st["h2d_bytes"],
                "d2h_bytes_per_step": 4 + st["d2h_bytes"]},
        "gpu_launches": kernels,
        "step_breakdown_ms": {k: st[k] for k in ("step_ms", "gpu_compute_ms", "h2d_ms", "d2h_ms", "wait_weights_ms",
                                                 "visit_gap_ms", "host_pre_ms", "tail_grads_ms", "tail_adam_ms",
                                                 "tail_rest_ms", "adam_ms", "adam_tail_ms", "gemm_ms")},
        "losses": losses, "init_seconds": init_s,
        "device_memory": dev_mem,
    }
    # Host memory traffic of a step: every uploaded byte is read from the
    # pageable tile, written to pinned staging and read by the DMA; every
    # gradient byte is written by the DMA (and, through the slabs, read and
    # written again by the accumulator); Adam reads and writes 22 bytes per
    # parameter (BF16 w and g, FP32 m and v; w, m, v written back).
    host_bytes = (3 if args.staged_weights else 1) * st["h2d_bytes"] + (3 if args.slab_grads else 1) * st["d2h_bytes"] + 22 * n_params
    line["host_memory"] = {"bytes_per_step": host_bytes, "gbs_measured": host_bw,
                           "t_ms": 1e3 * host_bytes / (host_bw * 1e9),
                           "frac_of_step": host_bytes / (host_bw * 1e9) / (ms_step * 1e-3),
                           "method": "torch CPU copy of 2 GiB, read + write bytes, all cores"}
    line["clocks"] = clk.summary()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = {k: v for k, v in cpu_sample(s).items() if k not in ("layer_seconds", "sample_seconds")}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
