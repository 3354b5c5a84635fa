"""Benchmark of the Medusa tree-verify step at Llama-7B shape on one GB300.

Workload: a random-init 32-layer Llama-7B-shaped decoder (d=4096, 32 heads x 128, FFN 11008 SiLU-gated,
vocabulary 32000, RMSNorm, RoPE) with 4 Medusa heads and the synthetic 64-node / 41-path tree (the 63
highest-scoring rank paths, score prod_d 0.7^d * 0.5^rank), after a random 128-token prompt, greedy
acceptance. One step = one medusa_verify_step: candidates, the backbone over the 64 tree tokens, the LM head,
the posterior, the KV compaction and the Medusa heads. Weights are bf16 (14.4 GB, far above the 129 MB L2,
so every step streams them from HBM).

Arms:
  default            the library (this repository's CUDA kernels)
  --impl reference   the CPU oracle on the host cores, each step a bounded sample of the same workload

One JSON line on stdout (rank 0). Under torchrun (N > 1) every rank runs an independent replica (the step does
not shard), the timed region is bracketed by a barrier and the max over ranks is reported.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "verify steps/s (7B shape, 64-node tree)"
PROMPT_LEN = 128
TREE = dict(n_nodes=64, depth=4, topk=10)
FORCED_STEPS = 20  # forced-acceptance steps timed after the main run


def tree_choices(name):
    """The bench's tree: the synthetic 64-node tree (default) or the page's own 63 choices ("大模型推理 memory
    bandwidth bound (5) - Medusa", 二.2), both 64 nodes of depth 4 with top-10 heads."""
    if name == "page":
        with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tests", "golden", "page4_tree.json")) as f:
            return [tuple(c) for c in json.load(f)["medusa_choices"]]
    return synth.synthetic_tree_choices(TREE["n_nodes"], TREE["depth"], TREE["topk"])


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms while running; the sampler is started (and its
    first sample awaited) before the timed region, and only the samples taken inside it are summarised."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.rows, self.proc = index, [], None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.rows.append(parts)

    def ready(self, timeout=5.0):
        """Wait for the first sample (nvidia-smi takes a moment to start), then mark where the timed region begins."""
        t0 = time.time()
        while self.proc is not None and not self.rows and time.time() - t0 < timeout:
            time.sleep(0.01)
        self.mark = len(self.rows)
        return self

    def stop(self):
        """End of the timed region: later samples are ignored."""
        self.end = len(self.rows)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        lo = getattr(self, "mark", 0)
        hi = getattr(self, "end", len(self.rows))
        rows = self.rows[lo:hi] if hi > lo else self.rows[lo:lo + 1]
        self.rows = rows
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------------------------- CPU oracle sample

def sample_weights(seed=0, layers=2, device=None):
    """float64 host copies of the weights the oracle sample reads (generated on the GPU when there is one)."""
    dims = synth.LLAMA7B
    sub = synth.ModelDims(d=dims.d, n_layers=layers, n_heads=dims.n_heads, head_dim=dims.head_dim, ffn=dims.ffn,
                          vocab=dims.vocab, n_medusa=1)
    dev = device or ("cuda" if torch.cuda.is_available() else "cpu")
    names = {n for n, _ in synth.weight_names(sub)}
    w = {n: t.double().cpu().numpy() for n, t in synth.model_weights(sub, seed, torch.bfloat16, dev, names).items()}
    return sub, w


def oracle_sample(sub, w, seed=0, min_seconds=10.0, max_reps=20, tree_name="synthetic"):
    """Times the float64 oracle on a bounded sample of one 7B verify step.

    Sample: sub.n_layers of the 32 decoder layers over the 64 tree tokens at prefix 128, the LM head, the
    posterior, and 1 of the 4 Medusa heads on the accepted node, repeated until min_seconds of CPU work.
    Scaled to a full step as 32/layers x (decoder layers) + LM head + posterior + 4 x (one head).
    Returns (seconds per full step, sample description, wall seconds timed).
    """
    from oracle.model import Backbone, KVCache, medusa_heads
    from oracle.posterior import GREEDY, evaluate_posterior
    from oracle.tree import tree_buffers

    dims = synth.LLAMA7B
    layers = sub.n_layers
    tree = tree_buffers(tree_choices(tree_name), TREE["topk"])
    P = PROMPT_LEN
    toks = synth.prompt_tokens(seed, 64, dims.vocab, name="tree_tokens").numpy()
    no_lm = dict(w)
    no_lm["lm_head"] = w["lm_head"][:1]
    per, wall, reps = [], 0.0, 0
    while reps < max_reps and (wall < min_seconds or reps < 2):
        cache = KVCache(sub, P + 64)
        cache.data[:, :, :, :P] = synth.normal(seed, "kv_prefix", cache.data[:, :, :, :P].shape,
                                               dtype=torch.float64).numpy()
        t0 = time.perf_counter()
        h, _ = Backbone(sub, no_lm.__getitem__).forward(toks, P + tree["position_ids"], cache, P, tree["attn_mask"])
        t1 = time.perf_counter()
        logits = h @ w["lm_head"].T
        post = evaluate_posterior(logits, toks, tree["retrieve"], GREEDY)
        t2 = time.perf_counter()
        medusa_heads(w.__getitem__, 1, h[post["next_node"]])
        t3 = time.perf_counter()
        per.append((t1 - t0) * dims.n_layers / layers + (t2 - t1) + (t3 - t2) * dims.n_medusa)
        wall += t3 - t0
        reps += 1
    sample = (f"{layers} of 32 decoder layers over the 64 tree tokens at prefix {P}, the LM head, the posterior "
              f"and 1 of 4 Medusa heads of one 7B verify step in float64 ({reps} repetitions, {wall:.1f} s); "
              f"scaled to a full step")
    return statistics.median(per), sample, wall


# --------------------------------------------------------------------------------------------- GPU arm

def run_gpu(args, world, rank, local):
    import medusa_tree_speculative_verify_gb300 as mv
    torch.cuda.set_device(local)
    dims = synth.LLAMA7B
    w = mv.pack_model_weights(synth.packed_weights(dims, 0, torch.bfloat16, "cuda"), drop_source=True)
    model = mv.Model(dims, w)
    tree = mv.Tree(tree_choices(args.tree), TREE["topk"])
    n_steps_total = args.warmup + 7 * args.steps + 8
    s_max = PROMPT_LEN + (TREE["depth"] + 1) * n_steps_total + 64
    s_max = (s_max + 63) // 64 * 64
    sess = mv.Session(model, tree, s_max)
    prompt = synth.prompt_tokens(0, PROMPT_LEN, dims.vocab).to(torch.int32).cuda()
    prm = mv.AcceptParams(mv.GREEDY)
    stream = torch.cuda.current_stream()

    sess.prefill(prompt)
    for _ in range(args.warmup):  # eager warm-up steps
        sess.step(prm)
    torch.cuda.synchronize()
    sess.steps_graph(args.steps, prm)  # capture K steps into one CUDA graph + one warm replay
    torch.cuda.synchronize()
    st, code = mv.get_error()
    if st != 0:
        raise RuntimeError(f"device error word {code:#x}")

    # the decode state before the timed replay: the eager pass below restarts from it and must reach the same state
    snap_ws, snap_kv = sess.ws.clone(), sess.kv.clone()

    # ---- timed: K steps (one graph replay), inputs resident in HBM
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        clk.ready()
        start.record(stream)
        sess.steps_graph(args.steps, prm)
        end.record(stream)
        torch.cuda.synchronize()
        clk.stop()
    barrier(world)
    ms = max_over_ranks(start.elapsed_time(end), world)
    r = sess.read_result()
    len_graph = int(sess.cur_len.item())
    state_graph = (r, len_graph, sess.head_topk.clone(), sess.kv[:, :, :, :len_graph].clone())

    # ---- the same K steps as a graph with a CUDA event recorded around every launch: per-kernel device time
    # (the event nodes sit between kernels, so this pass runs without launch overlap; its total is reported)
    prof = mv.Profiler(sess)
    prof.enable()
    sess.steps_graph(args.steps, prm)  # capture the profiled graph + one replay
    torch.cuda.synchronize()
    prof.read()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    len_before = int(sess.cur_len.item())
    a.record(stream)
    sess.steps_graph(args.steps, prm)
    b.record(stream)
    torch.cuda.synchronize()
    per_kind = prof.read()
    mean_prefix = 0.5 * (len_before + int(sess.cur_len.item()))
    # candidates, embed, first QKV, per layer one projection chain (with the layer's attention inside it, or a
    # separate attention launch before it), posterior, KV compaction, heads x 2
    attn_launches = round(per_kind["attention"][1] / args.steps)
    launches_per_step = 1 + 1 + 1 + dims.n_layers + attn_launches + 1 + 1 + 2
    prof.disable()
    profiled_ms = a.elapsed_time(b)

    # ---- K eager steps without events from the same starting state, for comparison with the graph replay
    sess.ws.copy_(snap_ws)
    sess.kv.copy_(snap_kv)
    del snap_ws, snap_kv
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(args.steps):
        sess.step(prm)
    b.record(stream)
    torch.cuda.synchronize()
    eager_ms = a.elapsed_time(b)
    st, code = mv.get_error()
    if st != 0:
        raise RuntimeError(f"device error word {code:#x}")
    r = sess.read_result()
    len_eager = int(sess.cur_len.item())
    graph_equals_eager = (r == state_graph[0] and len_eager == state_graph[1]
                          and torch.equal(sess.head_topk, state_graph[2])
                          and torch.equal(sess.kv[:, :, :, :len_eager], state_graph[3]))
    if not graph_equals_eager:
        raise RuntimeError("the timed graph replay and the same steps run eagerly reached different decode states")
    del state_graph

    # ---- e2e: the host-buffer entry point (H2D seeds, step, D2H result + next seeds, stream sync per step)
    k = dims.n_medusa * TREE["topk"]
    seeds = torch.zeros(1 + k, dtype=torch.int32).pin_memory()
    seeds_next = torch.zeros(1 + k, dtype=torch.int32).pin_memory()
    res_host = torch.zeros(mv.RESULT_INTS, dtype=torch.int32).pin_memory()
    seeds[0] = int(r["next_root"])
    seeds[1:] = sess.head_topk.reshape(-1).cpu()
    sess.step_host(prm, seeds, res_host, seeds_next)  # untimed: captures the host step's graph
    seeds.copy_(seeds_next)
    torch.cuda.synchronize()
    tok_e2e = 0
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sess.step_host(prm, seeds, res_host, seeds_next)
        seeds.copy_(seeds_next)
        tok_e2e += int(res_host[4])
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    barrier(world)

    # ---- forced acceptance: the heads' rank-0 candidates replaced by the model's own greedy continuation, so
    # every step accepts the whole depth (greedy Medusa output = greedy AR output), through the same host-buffer
    # entry point as e2e. The continuation comes from plain steps from the same state, which is then restored.
    depth = tree.depth
    snap_ws, snap_kv = sess.ws.clone(), sess.kv.clone()
    greedy = []
    while len(greedy) < (depth + 1) * FORCED_STEPS + depth + 2:
        sess.step(prm)
        greedy += sess.read_result()["tokens"]
    sess.ws.copy_(snap_ws)
    sess.kv.copy_(snap_kv)
    del snap_ws, snap_kv
    seeds[1:] = sess.head_topk.reshape(-1).cpu()
    torch.cuda.synchronize()
    pos, forced_ok, forced_full, forced_tok = 0, True, True, 0
    t0 = time.perf_counter()
    for _ in range(FORCED_STEPS):
        seeds[0] = greedy[pos]
        for h in range(dims.n_medusa):  # rank 0 of head h: the token h + 1 places after the root
            seeds[1 + h * TREE["topk"]] = greedy[pos + 1 + h]
        sess.step_host(prm, seeds, res_host, seeds_next)
        got = mv.result_dict(res_host)["tokens"]
        forced_ok &= got == greedy[pos: pos + len(got)]  # the emitted tokens are the greedy stream
        forced_full &= len(got) == depth + 1
        pos += len(got)
        forced_tok += len(got)
        seeds.copy_(seeds_next)
    forced_s = max_over_ranks(time.perf_counter() - t0, world)

    steps_per_s = args.steps / (ms / 1e3) * world
    tokens_per_step = tok_e2e / args.steps
    peak, peak_kind = peaks()
    gb = gemm_bytes(dims, TREE["n_nodes"])
    if attn_launches == 0:  # each layer's attention runs inside its chain: its bytes are the chain's too
        gb["gemm_chain"] += attention_bytes(dims, TREE["n_nodes"], mean_prefix)
    g_ms_prof = sum(per_kind[k][0] for k in gb)
    g_n = sum(per_kind[k][1] for k in gb)
    g_bytes = sum(gb[k] * per_kind[k][1] for k in gb)
    # The projection launches' time inside the timed replay: its ms per step times their share of the kernel time
    # in the profiled replay (events between launches there serialise the kernels and add a few us to each, so its
    # per-launch durations overstate; the share is what it measures well). The profiled figure is kept beside.
    share = g_ms_prof / max(sum(v[0] for v in per_kind.values()), 1e-9)
    g_ms = ms * share
    achieved = g_bytes / (g_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": "gemm_kernel (tcgen05 projections; per layer one launch of the layer's "
                                          "tree attention, O, gate/up, down and the next QKV, plus the first QKV)",
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak, "peak_kind": peak_kind,
                "traffic": GEMM_TRAFFIC_PER_ALGORITHMIC_BYTE * g_bytes / max(g_n, 1),
                "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of one chain launch with its "
                                  "layer's attention (profiles/gemm_kernel_fused_chain_7b_layer_t64.md), scaled to the "
                                  "step's average projection launch by its algorithmic bytes",
                "algorithmic_bytes_per_launch": g_bytes / max(g_n, 1),
                "avg_launch_us": g_ms * 1e3 / max(g_n, 1),
                "avg_launch_us_source": "timed graph replay x the projection launches' share of the kernel time "
                                        "in a replay with CUDA events around every launch",
                "share_of_step": share,
                "avg_launch_us_profiled": g_ms_prof * 1e3 / max(g_n, 1),
                "per_kind": {k: {"launches_per_step": c / args.steps, "ms_per_step": ms / args.steps,
                                 **({"gbs": gb[k] * c / (ms / 1e3) / 1e9} if k in gb and ms > 0 else {})}
                             for k, (ms, c) in per_kind.items()}}
    step_bytes = weight_bytes(dims)
    line = {
        "metric": METRIC, "value": steps_per_s, "unit": "steps/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (random-init weights, random prompt)",
        "config": {"workload": "Llama-7B shape (32 layers, d 4096, 32x128 heads, FFN 11008, vocab 32000) + 4 Medusa "
                               "heads, " + ("the page's own 63-choice (64-node, 42-path) tree" if args.tree == "page"
                                            else "synthetic 64-node/41-path tree") +
                               ", 128-token prompt, greedy verify step",
                   "tree_nodes": 64, "prompt": PROMPT_LEN, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (14.4 GB of weights streamed per step)"},
        "tokens_per_s": steps_per_s * tokens_per_step, "tokens_per_step": tokens_per_step,
        "forced_acceptance": {"steps": FORCED_STEPS, "tokens_per_step": forced_tok / FORCED_STEPS,
                              "e2e_tokens_per_s": forced_tok * world / forced_s,
                              "e2e_steps_per_s": FORCED_STEPS * world / forced_s,
                              "tokens_equal_greedy_stream": bool(forced_ok),
                              "all_steps_accept_the_whole_depth": bool(forced_full)},
        "step_hbm_gbs": step_bytes / (ms / args.steps / 1e3) / 1e9,
        "e2e": {"value": args.steps * world / e2e_s, "unit": "steps/s", "h2d_bytes_per_step": 4 * (1 + k),
                "d2h_bytes_per_step": 4 * mv.RESULT_INTS + 4 * (1 + k)},
        "gpu_launches": launches_per_step * args.steps,
        "timing": {"graph_ms_per_step": ms / args.steps, "profiled_graph_ms_per_step": profiled_ms / args.steps,
                   "eager_ms_per_step": eager_ms / args.steps, "graph_equals_eager": graph_equals_eager},
        "roofline": roofline,
        "clocks": clk.summary(),
    }
    return line


# DRAM bytes (read + write) per algorithmic byte of the projection kernel, from the ncu capture of one chain launch
# with its layer's attention (7B shape: 414.6 MB measured for 420.2 MB algorithmic; the LM-head launch alone:
# 268.4 / 270.9 MB): the kernel reads every weight byte once, so the traffic of a launch scales with its bytes.
GEMM_TRAFFIC_PER_ALGORITHMIC_BYTE = 0.987


def gemm_bytes(dims, n):
    """Algorithmic HBM bytes of one launch of each projection: weights once, activations in and out once."""
    d, HD, F, V = dims.d, dims.n_heads * dims.head_dim, dims.ffn, dims.vocab
    b = {"gemm_qkv": 2 * 3 * HD * d + 2 * n * d + 2 * n * 3 * HD,
         "gemm_o": 2 * d * HD + 2 * n * HD + 4 * n * d * 2 + 2 * n * d,
         "gemm_gate_up": 2 * 2 * F * d + 2 * n * d + 2 * n * F,
         "gemm_down": 2 * d * F + 2 * n * F + 4 * n * d * 2 + 2 * n * d,
         "gemm_lm": 2 * V * d + 2 * n * d + 4 * n * V}
    # one chain launch per layer: O, gate/up, down, then the next layer's QKV (the LM head after the last layer)
    L = dims.n_layers
    layer = b["gemm_o"] + b["gemm_gate_up"] + b["gemm_down"]
    b["gemm_chain"] = layer + ((L - 1) * b["gemm_qkv"] + b["gemm_lm"]) / L
    return b


def attention_bytes(dims, n, prefix):
    """Algorithmic bytes of one layer's tree attention: the prefix and tree keys and values once, q in, out."""
    HD = dims.n_heads * dims.head_dim
    return (prefix + n) * HD * 2 * 2 + 2 * n * HD * 2


MICRO = {  # name -> (M, K, n): projections of the 7B step, timed alone through mv_linear_bf16
    "lm_head": (32000, 4096, 64), "gate_up": (22016, 4096, 64), "down": (4096, 11008, 64),
    "qkv": (12288, 4096, 64), "o": (4096, 4096, 64),
}
MICRO_OTHER = ["heads_b1", "heads_b4", "heads_b16", "attn_p64", "attn_p512", "attn_p1024", "attn_p4096",
               "posterior_greedy", "posterior_typical", "kv_compact_acc4", "root_typical", "root_nucleus"]


def _time_launches(fn, steps, warmup, flush=True):
    """Median CUDA-event time (ms) of fn() on the current stream, L2 flushed before each by READING a 256 MB buffer
    (a flush by writing would leave dirty lines whose write-back then competes with the timed kernel's reads)."""
    buf = torch.ones(64 << 20, dtype=torch.float32, device="cuda") if flush else None
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    times = []
    for _ in range(steps):
        if buf is not None:
            buf.sum()
        torch.cuda._sleep(200000)  # keep the GPU busy while the launch is enqueued: no host latency in the event pair
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.median(times)


def run_micro_step2(steps, warmup):
    """Verify steps of a 2-layer model of the 7B shape (2.7 GB on the device: small enough for a full ncu capture of
    one projection-chain launch). Prefill of 128 tokens (2 chunks), `warmup` eager steps, then `steps` eager steps
    timed with CUDA events. Projection launches before the timed steps: 2 x (1 + 2) + warmup x (1 + 2)."""
    import dataclasses
    import medusa_tree_speculative_verify_gb300 as mv
    dims = dataclasses.replace(synth.LLAMA7B, n_layers=2)
    w = mv.pack_model_weights(synth.packed_weights(dims, 0, torch.bfloat16, "cuda"), drop_source=True)
    model = mv.Model(dims, w)
    tree = mv.Tree(tree_choices("synthetic"), TREE["topk"])
    sess = mv.Session(model, tree, 1024)
    sess.prefill(synth.prompt_tokens(0, PROMPT_LEN, dims.vocab).to(torch.int32).cuda())
    prm = mv.AcceptParams(mv.GREEDY)
    for _ in range(warmup):
        sess.step(prm)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        sess.step(prm)
    b.record()
    torch.cuda.synchronize()
    st, code = mv.get_error()
    if st != 0:
        raise RuntimeError(f"device error word {code:#x}")
    return {"micro": "step_2layers", "ms_per_step": a.elapsed_time(b) / steps,
            "gemm_launches_before_timed": 2 * (1 + dims.n_layers) + warmup * (1 + dims.n_layers)}


def run_micro_other(name, steps, warmup):
    """One standalone kernel of the path at the sizes of its workload; GB/s of its algorithmic bytes."""
    import medusa_tree_speculative_verify_gb300 as mv
    peak, kind = peaks()
    ws = lambda n: torch.zeros(max(n, 16), dtype=torch.uint8, device="cuda")
    tree = mv.Tree(synth.synthetic_tree_choices(64, 4, 10), 10)
    if name.startswith("heads_b"):
        B, d, K, V = int(name[7:]), 4096, 4, 32000
        w1 = synth.normal(0, "w1", (K, d, d), 0.02, dtype=torch.bfloat16, device="cuda")
        w2 = synth.normal(0, "w2", (K, V, d), 0.02, dtype=torch.bfloat16, device="cuda")
        wl = synth.normal(0, "lm", (V, d), 0.02, dtype=torch.bfloat16, device="cuda")
        h = synth.normal(0, "h", (B, d), 1.0, dtype=torch.bfloat16, device="cuda")
        oi = torch.empty(B, K, 10, dtype=torch.int32, device="cuda")
        ov = torch.empty(B, K, 10, dtype=torch.float32, device="cuda")
        root = torch.empty(B, dtype=torch.int32, device="cuda")
        w = ws(mv.medusa_heads_topk_workspace(B, d, K, V, 10))
        fn = lambda: mv.medusa_heads_topk(h, w1, w2, 10, oi, ov, w_lm=wl, out_root=root, workspace=w)
        nbytes = 2 * (K * d * d + K * V * d + V * d) + 2 * B * d
    elif name.startswith("attn_p"):
        P, H, D = int(name[6:]), 32, 128
        n = tree.n_nodes
        q = synth.normal(0, "q", (n, H, D), dtype=torch.bfloat16, device="cuda")
        k = synth.normal(0, "k", (H, P + n, D), dtype=torch.bfloat16, device="cuda")
        v = synth.normal(0, "v", (H, P + n, D), dtype=torch.bfloat16, device="cuda")
        out = torch.empty_like(q)
        w = ws(mv.tree_attention_workspace(H, D, P + n, n))
        fn = lambda: mv.tree_attention(q, k, v, P, tree, D ** -0.5, out, w)
        nbytes = (P + n) * H * D * 2 * 2 + 2 * n * H * D * 2
    elif name.startswith("posterior"):
        mode = mv.TYPICAL if name.endswith("typical") else mv.GREEDY
        path = [int(x) for x in tree.retrieve[0] if x >= 0]
        toks, logits = synth.planted_tokens_and_logits(0, tree.n_nodes, 32000, path, len(path) - 1)
        logits, toks = logits.cuda(), torch.as_tensor(toks, dtype=torch.int32, device="cuda")
        out = torch.empty(mv.RESULT_INTS, dtype=torch.int32, device="cuda")
        w = ws(mv.evaluate_posterior_workspace(tree.n_nodes))
        prm = mv.AcceptParams(mode, 0.7, 0.09, 0.3)
        fn = lambda: mv.evaluate_posterior(logits, toks, tree, prm, out, w)
        nbytes = tree.n_nodes * 32000 * 4
    elif name.startswith("root_"):  # one stochastic root draw from a 32000-logit row (T 0.7, top_p 0.8)
        mode = mv.ROOT_TYPICAL if name.endswith("typical") else mv.ROOT_NUCLEUS
        row = synth.normal(0, "root_row", (32000,), 2.0, device="cuda")
        out = torch.empty(1, dtype=torch.int32, device="cuda")
        prm = mv.RootParams(mode, 0.7, 0.09, 0.3, 0.8, key=1)
        fn = lambda: mv.sample_root(row, prm, 0, out)
        nbytes = 32000 * 4
    else:  # kv_compact_acc4: 32 layers x 32 heads x 128, prefix 1024, path of 5 nodes
        kv = synth.kv_cache(0, (32, 2, 32, 1088, 128), device="cuda")
        r = mv.PosteriorResult()
        r.acc, r.n_tokens = 4, 5
        for j, nd in enumerate([0, 1, 11, 34, 57]):
            r.nodes[j] = nd
        res = torch.tensor(np.frombuffer(bytes(r), dtype=np.int32).copy(), device="cuda")
        cur = torch.zeros(1, dtype=torch.int32, device="cuda")
        fn = lambda: mv.kv_compact(kv, 1024, res, cur)
        nbytes = 2 * 5 * 32 * 2 * 32 * 128 * 2
    ms = _time_launches(fn, steps, warmup)
    st, code = mv.get_error()
    if st != 0:
        raise RuntimeError(f"device error word {code:#x}")
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"micro": name, "median_us": ms * 1e3, "algorithmic_bytes": nbytes, "gbs": gbs, "frac": gbs / peak,
            "peak": peak, "peak_kind": kind, "l2": "flushed (256 MB read before each launch)"}


def run_micro(name, steps, warmup):
    """The projection kernel alone on one shape: HBM GB/s of weights + activations per launch (CUDA events)."""
    import medusa_tree_speculative_verify_gb300 as mv
    M, K, n = MICRO[name]
    w = synth.normal(1, "w", (M, K), 0.02, dtype=torch.bfloat16, device="cuda")
    wp = mv.pack_weight(w, 128)
    x = synth.normal(2, "x", (n, K), 1.0, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(n, M, dtype=torch.float32, device="cuda")
    ws = torch.zeros(mv.linear_bf16_workspace(), dtype=torch.uint8, device="cuda")
    nbytes = 2 * M * K + 2 * n * K + 4 * n * M
    peak, kind = peaks()
    ms_packed = _time_launches(lambda: mv.linear_bf16_packed(wp, M, K, x, out, ws), steps, warmup)
    ms_rowmajor = _time_launches(lambda: mv.linear_bf16(w, x, out, ws), steps, warmup)
    gbs = nbytes / (ms_packed / 1e3) / 1e9
    return {"micro": name, "M": M, "K": K, "n": n, "median_us": ms_packed * 1e3, "gbs": gbs, "frac": gbs / peak,
            "rowmajor_us": ms_rowmajor * 1e3, "rowmajor_gbs": nbytes / (ms_rowmajor / 1e3) / 1e9,
            "peak": peak, "peak_kind": kind, "l2": "flushed (256 MB read before each launch)", "layout": "packed"}


def run_sweep_nodes(sizes, steps, warmup):
    """Verify-step speed against the number of tree nodes (candidate tokens): the synthetic tree's n - 1
    highest-scoring paths for each n, the same 7B-shape model, K steps as one graph replay after a 128-token
    prompt. One JSON line per size. (The acceleration side of the trade-off, tokens accepted per step, needs
    trained heads; with random weights almost nothing is accepted, so only the cost side is measured.)"""
    import medusa_tree_speculative_verify_gb300 as mv
    dims = synth.LLAMA7B
    w = mv.pack_model_weights(synth.packed_weights(dims, 0, torch.bfloat16, "cuda"), drop_source=True)
    model = mv.Model(dims, w)
    prompt = synth.prompt_tokens(0, PROMPT_LEN, dims.vocab).to(torch.int32).cuda()
    prm = mv.AcceptParams(mv.GREEDY)
    stream = torch.cuda.current_stream()
    wb = weight_bytes(dims)
    for n in sizes:
        tree = mv.Tree(synth.synthetic_tree_choices(n, TREE["depth"], TREE["topk"]), TREE["topk"])
        s_max = (PROMPT_LEN + (TREE["depth"] + 1) * (warmup + 2 * steps + 2) + 64 + 63) // 64 * 64
        sess = mv.Session(model, tree, s_max)
        sess.prefill(prompt)
        for _ in range(warmup):
            sess.step(prm)
        sess.steps_graph(steps, prm)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(0) as clk:
            clk.ready()
            a.record(stream)
            sess.steps_graph(steps, prm)
            b.record(stream)
            torch.cuda.synchronize()
            clk.stop()
        ms = a.elapsed_time(b) / steps
        st, code = mv.get_error()
        if st != 0:
            raise RuntimeError(f"device error word {code:#x}")
        print(json.dumps({"sweep": "tree_nodes", "n_nodes": n, "n_paths": tree.n_paths, "depth": tree.depth,
                          "steps": steps, "ms_per_step": ms, "steps_per_s": 1e3 / ms,
                          "weight_gbs": wb / (ms / 1e3) / 1e9, "clocks": clk.summary()}), flush=True)
        del sess, tree


def run_sweep_batch(batches, steps, warmup, tree_name):
    """Verify steps of B independent sequences per session (one backbone pass for all B trees per step): one JSON
    line per B with the step time and the sequence-steps per second. Each sequence has its own 128-token prompt."""
    import medusa_tree_speculative_verify_gb300 as mv
    dims = synth.LLAMA7B
    w = mv.pack_model_weights(synth.packed_weights(dims, 0, torch.bfloat16, "cuda"), drop_source=True)
    model = mv.Model(dims, w)
    tree = mv.Tree(tree_choices(tree_name), TREE["topk"])
    prm = mv.AcceptParams(mv.GREEDY)
    stream = torch.cuda.current_stream()
    for B in batches:
        s_max = (PROMPT_LEN + (TREE["depth"] + 1) * (warmup + 2 * steps + 2) + 64 + 63) // 64 * 64
        sess = mv.Session(model, tree, s_max, batch=B)
        for b in range(B):
            sess.prefill_seq(b, synth.prompt_tokens(b, PROMPT_LEN, dims.vocab).to(torch.int32).cuda())
        for _ in range(warmup):
            sess.step(prm)
        sess.steps_graph(steps, prm)
        torch.cuda.synchronize()
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(0) as clk:
            clk.ready()
            a.record(stream)
            sess.steps_graph(steps, prm)
            b_.record(stream)
            torch.cuda.synchronize()
            clk.stop()
        ms = a.elapsed_time(b_) / steps
        # per-kind device time per step from a replay with an event pair around every launch
        prof = mv.Profiler(sess)
        prof.enable()
        sess.steps_graph(steps, prm)
        torch.cuda.synchronize()
        prof.read()
        sess.steps_graph(steps, prm)
        torch.cuda.synchronize()
        per_kind = {k: round(1e3 * v[0] / steps, 1) for k, v in prof.read().items() if v[1]}
        prof.disable()
        st, code = mv.get_error()
        if st != 0:
            raise RuntimeError(f"device error word {code:#x}")
        print(json.dumps({"sweep": "batch", "batch": B, "n_nodes": tree.n_nodes, "steps": steps, "ms_per_step": ms,
                          "steps_per_s": 1e3 / ms, "sequence_steps_per_s": B * 1e3 / ms,
                          "profiled_us_per_step_by_kind": per_kind, "clocks": clk.summary()}), flush=True)
        del sess


def weight_bytes(dims):
    d, HD, F, V, K, L = dims.d, dims.n_heads * dims.head_dim, dims.ffn, dims.vocab, dims.n_medusa, dims.n_layers
    per_layer = 2 * (3 * HD * d + d * HD + 2 * F * d + d * F)
    return L * per_layer + 2 * V * d + 2 * K * (d * d + V * d)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tree", default="synthetic", choices=["synthetic", "page"],
                    help="the tree of the verify step: the synthetic 64-node tree or the page's own 63 choices")
    ap.add_argument("--micro", choices=sorted(MICRO) + MICRO_OTHER + ["step_2layers"],
                    help="time one kernel alone and exit")
    ap.add_argument("--sweep-nodes", default=None,
                    help="comma-separated tree sizes (2..256): time the verify step per size and exit")
    ap.add_argument("--sweep-batch", default=None,
                    help="comma-separated batch sizes (1..4): time the batched verify step per size and exit")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.sweep_nodes:
        run_sweep_nodes([int(x) for x in args.sweep_nodes.split(",")], args.steps, args.warmup)
        return
    if args.sweep_batch:
        run_sweep_batch([int(x) for x in args.sweep_batch.split(",")], args.steps, args.warmup, args.tree)
        return
    if args.micro:
        if args.micro == "step_2layers":
            print(json.dumps(run_micro_step2(args.steps, args.warmup)))
            return
        fn = run_micro if args.micro in MICRO else run_micro_other
        print(json.dumps(fn(args.micro, args.steps, args.warmup)))
        return

    if args.impl == "reference":
        if rank != 0:
            return
        sub, w = sample_weights()
        oracle_sample(sub, w, min_seconds=0.0, max_reps=max(1, min(args.warmup, 2)), tree_name=args.tree)   # warm-up
        per_step, sample, _ = oracle_sample(sub, w, min_seconds=0.0, max_reps=max(2, min(args.steps, 20)), tree_name=args.tree)
        v = 1.0 / per_step
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 / v, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": "Llama-7B shape + 4 Medusa heads, synthetic 64-node tree, 128-token prompt"},
                "cpu_baseline": {"value": v, "unit": "steps/s", "cores": os.cpu_count(), "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    line = run_gpu(args, world, rank, local)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            sub, w = sample_weights()
            per_step, sample, wall = oracle_sample(sub, w, tree_name=args.tree)
            line["cpu_baseline"] = {"value": 1.0 / per_step, "unit": "steps/s", "cores": os.cpu_count(),
                                    "kind": "oracle", "sample": sample, "sample_wall_s": wall}
        print(json.dumps(line))


if __name__ == "__main__":
    main()
