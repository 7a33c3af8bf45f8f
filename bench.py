#!/usr/bin/env python3
"""Benchmark of the compressed sparse attention layer core on GB300.

One step = one pass of the whole layer (attn_v41_forward: projections, RoPE, fp8 window rows, ring,
indexer scores, top-k, sparse attention with the sink, grouped output) for one batch of the
workload, inputs resident in HBM.  The metric is decode tokens per second per layer; the line
also reports the sparse-attention + indexer + top-k HBM bandwidth against 8 TB/s and the measured
copy bandwidth, the dominant kernel's roofline, an end-to-end figure through the host-buffer entry
point, and the CPU oracle timed on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl csa|reference]

Timing: W untimed steps, then K steps captured once as a CUDA graph and replayed, each bracketed
by CUDA events on the launching stream; L2 is flushed (a 512 MiB memset) between timed steps and
outside the event pair.  N > 1 (torchrun): every rank runs the full workload on its own GPU
(replicas, weak scaling, no collective on the data path); value = all ranks' tokens / the slowest
rank's time.
"""
import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s per layer; sparse_attn+indexer HBM GB/s vs 8 TB/s (1×GB300)"
DEFAULT_WORKLOAD = "reindex_decode_r2"
NOMINAL_HBM_GBS = 8000.0
# ncu dram__bytes_read.sum + dram__bytes_write.sum of one forward's projection launches (proj x, proj
# qr, wo_a, wo_b), copied from the ncu capture summarised in the file below (not measured in this
# run); set to None whenever those kernels change after the capture
GEMM_TRAFFIC_SOURCE = "ncu capture, profiles/k_gemm_tc_projections_all_workloads.md"
GEMM_TRAFFIC_BYTES = {
    "reindex_decode_r2": (19072000 + 0) + (94519040 + 151808) + (69267712 + 6656) + (84563712 + 164608),
    "longctx_decode_r4": (19400960 + 0) + (94602496 + 142592) + (71365888 + 62208) + (85174272 + 237056),
    "ratio0_decode": (18744320 + 0) + (84032000 + 179712) + (69281792 + 12800) + (84606208 + 143872),
    # (prefill: wo_b's whole waves, its split last wave and their sum are three launches)
    "prefill_r4": (68499712 + 5202944) + (104963840 + 251502336) + (428238080 + 50825728) +
                  (353134848 + 29880064) + (71337728 + 114688) + (16785152 + 0),
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="csa", choices=["csa", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-extra", action="store_true",
                   help="skip the long-context and prefill figures the default workload's line adds")
    return p.parse_args()


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


# --------------------------------------------------------------------------------------- inputs

def build_inputs(wl, rank=0):
    """Seeded numpy inputs of the workload (bf16 as uint16 bit patterns)."""
    from csa_inputs import activations, candidate_mask, latent_cache, positions, ring_rows, weights
    g = wl.geom
    B, T, start = wl.batch, wl.tokens, wl.start_pos
    layers = []
    for l in range(wl.layers):
        layers.append(weights(g, with_indexer=wl.is_index_source, seed_base=1000 + 100 * l))
    x = activations(g, B, T, seed_base=1000 + 7 * rank)
    ring = ring_rows(g, B) if start else np.zeros((B, g.window, g.head_dim), np.uint16)
    shared = None
    if wl.ratio:
        L = wl.compress_len
        Z, KI = latent_cache(g, B, L)
        pos = positions(B, T, start)
        cand = None
        if wl.uses_candidates:
            cand = candidate_mask(B * T, pos, wl.ratio, L, g.cand_block, -(-L // g.cand_block), wl.cand_keep, 1015)
        shared = dict(Z=Z, KI=KI, L=L, cand=cand)
    return layers, x, ring, shared


def algorithmic_bytes(wl, shared_np, idx_counts):
    """Per-step algorithmic bytes of the sparse attention, indexer and top-k (all layers), from the
    workload's selection sizes: q and output once, each gathered row once, each candidate key once."""
    g = wl.geom
    H, hd, NT = g.n_heads, g.head_dim, wl.batch * wl.tokens
    rows, n_valid = idx_counts
    attn = NT * (H * hd * 2 * 2 + (g.window + (g.index_topk if wl.ratio else 0)) * 4) + rows * hd * 2
    idx = topk = 0
    if wl.ratio and wl.is_index_source:
        cw = 0 if shared_np["cand"] is None else shared_np["cand"].shape[1]
        idx = NT * (g.index_heads * g.index_hd * 2 + g.index_heads * 4 + cw) + n_valid * (g.index_hd * 2 + 4)
        topk = NT * (cw + g.index_topk * 4) + n_valid * 4
    return attn * wl.layers, idx * wl.layers, topk * wl.layers


def projection_bytes(wl):
    """Per-step algorithmic bytes of each projection stage (all layers), bf16: its weights [out, in]
    read once, its input activations read once and its outputs written once."""
    g = wl.geom
    M = wl.batch * wl.tokens
    isrc = bool(wl.ratio and wl.is_index_source)
    gw = g.n_heads * g.head_dim // g.groups
    # (weights [out, in], activation width read, output width written) of one layer
    stages = {
        "proj x": ([(g.q_rank, g.dim), (g.head_dim, g.dim)] + ([(g.index_heads, g.dim)] if isrc else []), g.dim,
                   g.q_rank + g.head_dim + (g.index_heads if isrc else 0)),
        "proj qr": ([(g.n_heads * g.head_dim, g.q_rank)] + ([(g.index_heads * g.index_hd, g.q_rank)] if isrc else []),
                    g.q_rank, g.n_heads * g.head_dim + (g.index_heads * g.index_hd if isrc else 0)),
        "wo_a": ([(g.groups * g.o_rank, gw)], g.n_heads * g.head_dim, g.groups * g.o_rank),
        "wo_b": ([(g.dim, g.groups * g.o_rank)], g.groups * g.o_rank, g.dim),
    }
    return {n: wl.layers * 2 * (sum(a * b for a, b in ws_) + M * xin + M * yout) for n, (ws_, xin, yout) in stages.items()}


def projection_flops(wl):
    """Per-step algorithmic flops of each projection stage (all layers): 2 x tokens x out x in."""
    g = wl.geom
    M = wl.batch * wl.tokens
    isrc = bool(wl.ratio and wl.is_index_source)
    gw = g.n_heads * g.head_dim // g.groups
    ws = {
        "proj x": [(g.q_rank, g.dim), (g.head_dim, g.dim)] + ([(g.index_heads, g.dim)] if isrc else []),
        "proj qr": [(g.n_heads * g.head_dim, g.q_rank)] + ([(g.index_heads * g.index_hd, g.q_rank)] if isrc else []),
        "wo_a": [(g.groups * g.o_rank, gw)],
        "wo_b": [(g.dim, g.groups * g.o_rank)],
    }
    return {n: wl.layers * 2.0 * M * sum(a * b for a, b in w) for n, w in ws.items()}


def selection_counts(wl, shared_np):
    """(gathered rows, valid compressed positions) summed over the batch's queries."""
    g = wl.geom
    B, T, start = wl.batch, wl.tokens, wl.start_pos
    rows = n_valid = 0
    for r in range(B * T):
        t = r % T
        p = start + t
        rows += min(p + 1, g.window)
        if wl.ratio:
            limit = min((p + 1) // wl.ratio, shared_np["L"])
            if shared_np["cand"] is not None:
                c = shared_np["cand"][r]
                nv = sum(min(g.cand_block, limit - b * g.cand_block) for b in range(len(c))
                         if c[b] and b * g.cand_block < limit)
            else:
                nv = limit
            n_valid += nv
            rows += min(nv, g.index_topk)
    return rows, n_valid


# --------------------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.dev = device_index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                                       "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        time.sleep(0.25)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [s.strip() for s in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.f.name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------------------- CPU oracle

def oracle_sample(wl, layers, x, ring, shared_np, seqs, tok_rows=None):
    """One oracle layer pass (all layers of the workload) over a subset of the batch."""
    import oracle as orc
    g = wl.geom
    gd = g.as_dict()
    T, start = wl.tokens, wl.start_pos
    tab = orc.rope_table(g.rope_dim, g.max_seq, g.compress_rope_theta if wl.ratio else g.rope_theta,
                         g.orig_seq if wl.ratio else 0, g.rope_factor, g.beta_fast, g.beta_slow)
    role = dict(ratio=wl.ratio, is_index_source=int(wl.is_index_source), uses_candidates=int(wl.uses_candidates))
    ntok = 0
    for b in seqs:
        ring_b = orc.act_quant(ring[b:b + 1])[0] if start else ring[b:b + 1].copy()
        sh = None
        if shared_np is not None:
            sh = dict(compress_kv=shared_np["Z"][b:b + 1], index_k=shared_np["KI"][b:b + 1], compress_len=shared_np["L"],
                      topk_idxs=np.zeros((T, g.index_topk), np.int32))
            if shared_np["cand"] is not None:
                sh["candidates"] = shared_np["cand"][b * T:(b + 1) * T]
        mask = None
        if tok_rows is not None:
            mask = np.zeros(T, np.uint8)
            mask[tok_rows] = 1
        for w in layers:
            orc.attn_forward(gd, role, w, ring_b, x[b:b + 1], start, tab, sh, tok_mask=mask, debug=False)
        ntok += T if tok_rows is None else len(tok_rows)
    return ntok


def cpu_baseline(wl, layers, x, ring, shared_np, target_s):
    import oracle as orc
    orc.build()
    B, T = wl.batch, wl.tokens
    tok_rows = None if T == 1 else list(range(0, T, max(1, T // 8)))[:8]
    t0 = time.perf_counter()
    ntok, nseq, b = 0, 0, 0
    while True:
        ntok += oracle_sample(wl, layers, x, ring, shared_np, [b % B], tok_rows)
        nseq += 1
        b += 1
        if time.perf_counter() - t0 >= target_s or nseq >= 64 * B:
            break
    dt = time.perf_counter() - t0
    what = "%d sequence(s) x %s of the %s workload, %d layer(s) each" % (
        nseq, "1 decode token" if T == 1 else "%d sampled queries of the %d-token chunk" % (len(tok_rows), T),
        wl.name, wl.layers)
    return {"value": ntok / dt, "unit": "tokens/s", "cores": orc.num_threads(), "kind": "oracle", "sample": what,
            "seconds": round(dt, 3)}


# --------------------------------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    if rank != 0:
        return
    from csa_inputs import WORKLOADS
    import oracle as orc
    orc.build()
    wl = WORKLOADS[args.workload]
    layers, x, ring, shared_np = build_inputs(wl)
    T = wl.tokens
    tok_rows = None if T == 1 else list(range(0, T, max(1, T // 4)))[:4]
    seq_per_step = 1
    for i in range(args.warmup):
        oracle_sample(wl, layers, x, ring, shared_np, [i % wl.batch], tok_rows)
    times, ntok = [], 0
    for i in range(args.steps):
        t0 = time.perf_counter()
        ntok += oracle_sample(wl, layers, x, ring, shared_np, [(i * seq_per_step) % wl.batch], tok_rows)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = ntok / total
    sample = "per step: %s of one sequence of the %s workload, %d layer(s)" % (
        "1 decode token" if T == 1 else "%d sampled queries" % len(tok_rows), wl.name, wl.layers)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": wl.name, "batch": wl.batch, "tokens": wl.tokens,
                                            "start_pos": wl.start_pos, "ratio": wl.ratio, "layers": wl.layers},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": orc.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------------------- GPU arm

def max_over_ranks(ms, dist, device):
    """The timed region's length is the slowest rank's (every rank gets it back)."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, tokens_per_step, layers, steps, total_ms):
    """Whole-job throughput: every rank processes its own full batch (weak scaling)."""
    return world * tokens_per_step * layers * steps / (total_ms / 1000.0)


class Session:
    """One workload's device inputs, context and step on this rank's GPU."""

    def __init__(self, wl, rank, fp8_wo_a=False):
        import torch
        import compressed_sparse_attention_attn_gb300 as csa
        self.wl = wl
        g = wl.geom
        B, T, start, K = wl.batch, wl.tokens, wl.start_pos, g.index_topk
        self.np = build_inputs(wl, rank)
        layers_np, x_np, ring_np, sh_np = self.np
        if fp8_wo_a:
            # the grouped wo_a kept as e4m3 codes with one f32 scale per 128 x 128 tile (seeded storage)
            from csa_inputs import fp8_weight
            gw = g.n_heads * g.head_dim // g.groups
            layers_np = [dict(w) for w in layers_np]
            for l, w in enumerate(layers_np):
                w["wo_a_fp8"], w["wo_a_scale"] = fp8_weight((g.groups * g.o_rank, gw), 4100 + 100 * l)
                del w["wo_a"]

        def dev_bf16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

        self.ctx = csa.Context(g.as_dict())
        self.stream = torch.cuda.Stream()
        torch.cuda.set_stream(self.stream)
        self.role = dict(ratio=wl.ratio, is_index_source=int(wl.is_index_source),
                         uses_candidates=int(wl.uses_candidates))
        W = [{k: (dev_bf16(v) if v.dtype == np.uint16 else torch.from_numpy(v).cuda()) for k, v in w.items()}
             for w in layers_np]
        self.W = W
        self.lws = [csa.Context.layer_weights(w, self.role) for w in W]
        self.x = dev_bf16(x_np)
        self.out = torch.empty_like(self.x)
        self.rings = []
        for _ in range(wl.layers):
            r = dev_bf16(ring_np)
            if start:
                csa.act_quant(r)  # the ring holds fp8-rounded rows
            self.rings.append(r)
        self.shared = None
        if sh_np is not None:
            sel = torch.full((B * T, K), -1, dtype=torch.int32, device="cuda")
            cand = None if sh_np["cand"] is None else torch.from_numpy(sh_np["cand"]).cuda()
            self.shared = csa.Shared(dev_bf16(sh_np["Z"]), dev_bf16(sh_np["KI"]), sh_np["L"], sel, K, cand)
        self.flush_buf = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")

    def step(self):
        wl = self.wl
        for l in range(wl.layers):
            self.ctx.forward(None, self.role, self.rings[l], self.x, wl.start_pos, shared=self.shared, out=self.out,
                             lw=self.lws[l])

    def flush(self):
        self.flush_buf.zero_()

    def warm(self, n):
        import torch
        for _ in range(max(n, 3)):
            self.step()
        torch.cuda.synchronize()

    def capture(self):
        import torch
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=self.stream):
            self.step()
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()
        return graph

    def timed(self, graph, steps):
        """CUDA-event milliseconds of `steps` replays of graph, L2 flushed before each (outside the events)."""
        import torch
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for i in range(steps):
            self.flush()
            ev[i][0].record(self.stream)
            graph.replay()
            ev[i][1].record(self.stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]

    def stage_times(self, steps):
        """Per-step milliseconds of each stage (summed over the layers), from a captured step whose
        stages are bracketed by event-record nodes, replayed `steps` times with L2 flushed before each
        replay.  Falls back to eager traced forwards if the driver cannot time graph events."""
        import torch
        ctx = self.ctx
        acc = {}
        how = "graph replay (event-record nodes around each stage)"
        try:
            ctx.trace(True, append=True)
            graph = self.capture()
            for _ in range(steps):
                self.flush()
                graph.replay()
                for name, ms in ctx.trace_read():
                    acc[name] = acc.get(name, 0.0) + ms
            del graph
        except Exception:
            acc = {}
            how = "eager forwards (an event pair around each stage)"
            ctx.trace(True)
            for _ in range(steps):
                self.flush()
                for l in range(self.wl.layers):
                    ctx.forward(None, self.role, self.rings[l], self.x, self.wl.start_pos, shared=self.shared,
                                out=self.out, lw=self.lws[l])
                    for name, ms in ctx.trace_read():
                        acc[name] = acc.get(name, 0.0) + ms
        ctx.trace(False)
        torch.cuda.synchronize()
        return {k: v / steps for k, v in acc.items()}, how

    def close(self):
        import torch
        self.ctx.close()
        self.W = self.lws = self.x = self.out = self.rings = self.shared = self.flush_buf = None
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def attn_indexer_report(wl, sh_np, stage_ms, hbm_peak):
    counts = selection_counts(wl, sh_np)
    b_attn, b_idx, b_topk = algorithmic_bytes(wl, sh_np, counts)
    t_attn = stage_ms.get("sparse_attn", 0.0)
    # (short decode rows run scores and top-k as one kernel: its time counts as the indexer's)
    t_idx = stage_ms.get("index scores", 0.0) + stage_ms.get("index scores + topk", 0.0)
    t_topk = stage_ms.get("index topk", 0.0)
    ai_bytes = b_attn + b_idx + b_topk
    ai_ms = t_attn + t_idx + t_topk
    ai_gbs = ai_bytes / (ai_ms * 1e6) if ai_ms > 0 else None
    return {"bytes_per_step": int(ai_bytes), "ms_per_step": round(ai_ms, 5),
            "achieved_gbs": None if ai_gbs is None else round(ai_gbs, 1),
            "frac_of_8tbs": None if ai_gbs is None else round(ai_gbs / NOMINAL_HBM_GBS, 4),
            "frac_of_measured": None if ai_gbs is None else round(ai_gbs / hbm_peak, 4),
            "sparse_attn_ms": round(t_attn, 5), "index_scores_ms": round(t_idx, 5),
            "index_topk_ms": round(t_topk, 5), "gathered_rows": counts[0], "candidate_keys": counts[1]}


def scored_pairs(wl, sh_np):
    """Valid query-key pairs whose scores the selection reads: without a candidate mask, a query with
    at most index_topk valid positions takes all of them and its scores are not computed."""
    if sh_np["cand"] is not None:
        return selection_counts(wl, sh_np)[1]
    n = 0
    for r in range(wl.batch * wl.tokens):
        p = wl.start_pos + r % wl.tokens
        limit = min((p + 1) // wl.ratio, sh_np["L"]) if wl.ratio else 0
        if limit > wl.geom.index_topk:
            n += limit
    return n


def prefill_tensor_report(wl, sh_np, stage_ms, tflops_peak):
    """Algorithmic tensor work of the prefill's sparse attention (QK^T and PV over the gathered rows,
    4 H hd flops a row) and indexer scores (2 Hi dI flops per scored query-key pair: the pairs of the
    queries whose selection reads scores) over their times."""
    g = wl.geom
    rows, n_valid = selection_counts(wl, sh_np)
    f_attn = 4.0 * g.n_heads * g.head_dim * rows * wl.layers
    f_idx = 2.0 * g.index_heads * g.index_hd * scored_pairs(wl, sh_np) * wl.layers
    t_attn = stage_ms.get("sparse_attn", 0.0)
    t_idx = stage_ms.get("index scores", 0.0) + stage_ms.get("index scores + topk", 0.0)
    out = {}
    for name, f, t in (("sparse_attn", f_attn, t_attn), ("index_scores", f_idx, t_idx)):
        tf = f / (t * 1e9) if t > 0 else None
        out[name] = {"gflop": round(f / 1e9, 2), "ms": round(t, 5), "tflops": None if tf is None else round(tf, 1),
                     "frac_of_measured_bf16": None if tf is None else round(tf / tflops_peak, 4)}
    out["index_scores"]["gflop_all_valid_pairs"] = round(2.0 * g.index_heads * g.index_hd * n_valid * wl.layers / 1e9, 2)
    out["index_topk_ms"] = round(stage_ms.get("index topk", 0.0), 5)
    return out


def run_csa(args, rank, world, dist):
    import torch
    from csa_inputs import WORKLOADS

    dev = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(dev)
    wl = WORKLOADS[args.workload]
    g = wl.geom
    B, T, start = wl.batch, wl.tokens, wl.start_pos
    S = Session(wl, rank)
    ctx, stream = S.ctx, S.stream
    sh_np = S.np[3]

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    S.warm(args.warmup)
    launches_per_step = ctx.last_launches() * wl.layers
    graph = S.capture()

    # ---- timed region
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(dev)
    barrier()
    clocks.start()
    time.sleep(0.3)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        S.flush()
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
    barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = sum(step_ms)
    total_ms = max_over_ranks(total_ms, dist, "cuda")
    ms_per_step = total_ms / args.steps
    tokens_per_step = B * T  # per layer per rank
    value = job_tokens_per_s(world, tokens_per_step, wl.layers, args.steps, total_ms)

    # ---- per-stage kernel timing (replayed traced graph, flushed), for the roofline
    stage_ms, stage_how = S.stage_times(args.steps)
    lin_bytes = lin_flops = lin_ms = 0.0
    pflops = projection_flops(wl)
    for n, nbytes in projection_bytes(wl).items():
        if n in stage_ms:
            lin_bytes += nbytes
            lin_flops += pflops[n]
            lin_ms += stage_ms[n]
    peaks = measured_peaks()
    hbm_peak = peaks["hbm_gbs"] if peaks else 6800.0
    tflops_peak = peaks["bf16_tflops"] if peaks else 1900.0
    peak_src = "measured" if peaks else "fallback"
    traffic = GEMM_TRAFFIC_BYTES.get(wl.name)
    # the bound is whichever of the two floors is higher: the bytes at the copy bandwidth (few tokens,
    # weight streaming) or the flops at the bf16 GEMM rate (a prefill chunk's thousands of tokens)
    tensor_bound = lin_flops / (tflops_peak * 1e12) > lin_bytes / (hbm_peak * 1e9)
    if tensor_bound:
        achieved = lin_flops / (lin_ms * 1e9) if lin_ms > 0 else 0.0
        peak, unit, bound = tflops_peak, "TFLOP/s", "tensor"
    else:
        achieved = lin_bytes / (lin_ms * 1e6) if lin_ms > 0 else 0.0
        peak, unit, bound = hbm_peak, "GB/s", "hbm"
    roofline = {"kernel": "linear (the projections proj x, proj qr, wo_a, wo_b; all launches of one step)",
                "bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
                "frac": round(achieved / peak, 4),
                "traffic": None if traffic is None else traffic * wl.layers,
                "traffic_source": None if traffic is None else GEMM_TRAFFIC_SOURCE,
                "algorithmic_bytes": int(lin_bytes), "algorithmic_flops": int(lin_flops), "peak_source": peak_src,
                # of the traced stages' time (each stage bracketed by event records, so launches that
                # overlap in the untraced step do not here; their sum can exceed the untraced step)
                "share_of_traced_stages": round(lin_ms / sum(stage_ms.values()), 3) if stage_ms else None}

    # ---- end to end through the host-buffer entry point (pinned x in, out back to the host)
    x_host = S.x.cpu().pin_memory()
    out_host = torch.empty_like(x_host).pin_memory()

    def step_host():
        for l in range(wl.layers):
            ctx.forward_host(S.lws[l], S.rings[l], x_host, start, S.shared, out_host, B, T)

    for _ in range(2):
        step_host()
    torch.cuda.synchronize()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=stream):
        step_host()
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier()
    for i in range(args.steps):
        S.flush()
        ev2[i][0].record(stream)
        g2.replay()
        ev2[i][1].record(stream)
    barrier()
    e2e_ms = sum(a.elapsed_time(b) for a, b in ev2)
    e2e_ms = max_over_ranks(e2e_ms, dist, "cuda")
    e2e_value = job_tokens_per_s(world, tokens_per_step, wl.layers, args.steps, e2e_ms)
    io_bytes = wl.layers * B * T * g.dim * 2

    line = None
    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": wl.name, "batch": B, "tokens": T, "start_pos": start, "ratio": wl.ratio,
                           "compress_len": wl.compress_len, "layers": wl.layers,
                           "index_source": bool(wl.is_index_source), "candidates": bool(wl.uses_candidates),
                           "l2": "flushed between timed steps (512 MiB memset outside the events)",
                           "graph": "one step captured, replayed", "per_rank_batch": B},
                "attn_indexer": attn_indexer_report(wl, sh_np, stage_ms, hbm_peak),
                "stages_ms": {k: round(v, 5) for k, v in stage_ms.items()},
                "stage_timing": stage_how,
                "roofline": roofline,
                "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": io_bytes,
                        "d2h_bytes_per_step": io_bytes},
                "gpu_launches": launches_per_step * args.steps,
                "clocks": clk, "wall_s": round(wall, 4)}
    del graph, g2
    data = (wl, S.np[0], S.np[1], S.np[2], sh_np)
    S.close()

    # ---- the other configurations' figures of the metric's second part, timed in the same run: the
    # long-context decode's sparse attention + indexer + top-k bandwidth and the prefill chunk's
    # attention and indexer tensor throughput
    if line is not None and args.workload == DEFAULT_WORKLOAD and not args.no_extra:
        # the same decode step with the grouped wo_a kept in fp8 (e4m3 codes, one scale per 128 x 128 tile)
        Sf = Session(wl, rank, fp8_wo_a=True)
        Sf.warm(args.warmup)
        gf = Sf.capture()
        fms = sum(Sf.timed(gf, args.steps)) / args.steps
        del gf
        stf, how = Sf.stage_times(args.steps)
        gw = g.n_heads * g.head_dim // g.groups
        wbytes = g.groups * g.o_rank * gw + 4 * (-(-g.groups * g.o_rank // 128)) * (-(-gw // 128)) + \
            2 * B * T * (g.n_heads * g.head_dim + g.groups * g.o_rank)
        wo_ms = stf.get("wo_a", 0.0)
        line["fp8_wo_a"] = {"ms_per_step": round(fms, 5), "tokens_per_s": round(B * T * wl.layers / (fms / 1000.0), 1),
                            "wo_a_ms": round(wo_ms, 5), "wo_a_bytes": int(wbytes),
                            "wo_a_gbs": round(wbytes / (wo_ms * 1e6), 1) if wo_ms > 0 else None,
                            "wo_a_frac_of_measured": round(wbytes / (wo_ms * 1e6) / hbm_peak, 4) if wo_ms > 0 else None,
                            "stages_ms": {k: round(v, 5) for k, v in stf.items()}, "stage_timing": how,
                            "weights": "wo_a e4m3 codes + f32 scale per 128x128 tile (seeded); other weights bf16"}
        Sf.close()
        for name, key in (("longctx_decode_r4", "longctx_attn_indexer"), ("prefill_r4", "prefill_tensor")):
            wx = WORKLOADS[name]
            Sx = Session(wx, rank)
            Sx.warm(args.warmup)
            st, how = Sx.stage_times(max(3, min(args.steps, 10)))
            if name == "prefill_r4":
                rep = prefill_tensor_report(wx, Sx.np[3], st, tflops_peak)
            else:
                rep = attn_indexer_report(wx, Sx.np[3], st, hbm_peak)
            rep["workload"] = name
            rep["layers"] = wx.layers
            rep["stage_timing"] = how
            line[key] = rep
            Sx.close()
    return line, data


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist_
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist_.init_process_group("nccl")
        dist = dist_
    line, data = run_csa(args, rank, world, dist)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            wl, layers_np, x_np, ring_np, sh_np = data
            line["cpu_baseline"] = cpu_baseline(wl, layers_np, x_np, ring_np, sh_np, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
