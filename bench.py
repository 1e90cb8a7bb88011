"""Benchmark: greedy KV-cached generation through a BLOOM decoder stack on GB300.

One step = one whole generation of the workload: prefill of the B padded
prompts, then new_tokens - 1 decode steps (graph replays), the argmax fed back
on the device.  value = tokens/s = B * new_tokens / (time per step); the
pages' per-token cost is its inverse (wall time / (batch x tokens)).

The default workload is the 7b1-shaped stack (30 layers, h 4096, 32 heads,
vocab 250880) at batch 32, prompt 16, 100 greedy tokens.  The same line also
carries, as extra keys, the decode step at batch 1 / 8 / 64 / 128 of that
stack, its int8 weight-only form, and the 176B-layer-shaped stack (14 layers,
h 14336, 112 heads) at batch 1; each with its fraction of the HBM roofline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config 560m|7b1|7b1int8|176b14|block] [--batch B] [--no-extras]

Prints one JSON line (rank 0).  Under torchrun every rank runs its own replica
on its own GPU (sequences are independent; no collective on the data path).
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from bloom_decoder_token_gb300 import synth  # noqa: E402

METRIC = "decode ms/token & tokens/s (batch x tokens) and % of HBM roofline, 1 GB300"
UNIT = "tokens/s"
L2_BYTES = 129 * 2 ** 20
DEFAULT_CONFIG = "7b1"
DEFAULT_BATCH = {"7b1": 32, "7b1int8": 32}
SERIES_BATCHES = (1, 8, 32, 64, 128)   # decode-step series of the 7b1 stack


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def bf16_peak():
    """Dense bf16 tensor peak in TFLOP/s (the burst figure: prefill is timed
    launch by launch, seconds at most)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


# ------------------------------------------------------------------ byte model
def linear_shapes(sh: synth.Shape):
    h, F = sh.hidden, sh.ffn
    return {"qkv": (3 * h, h), "dense": (h, h), "up": (F, h), "down": (h, F)}


def weight_bytes(sh: synth.Shape) -> int:
    """Algorithmic bytes of all weights one decode step reads once."""
    h, V, L = sh.hidden, sh.vocab, sh.n_layer
    per = 0
    for N, K in linear_shapes(sh).values():
        per += N * K * (1 if sh.int8 else 2) + N * 2 + (N * 2 if sh.int8 else 0)   # W, bias, scales
    per += 4 * h * 2                                                               # 2 LayerNorms
    return L * per + V * h * 2 + 4 * h * 2                                         # + head E, ln_f, emb LN


def decode_step_bytes(sh: synth.Shape, B: int, keys: int) -> int:
    """Weights + KV read (keys slots, incl. the new one) + KV write + embedding rows."""
    h, L = sh.hidden, sh.n_layer
    kv_read = B * L * 2 * keys * h * 2
    kv_write = B * L * 2 * h * 2
    return weight_bytes(sh) + kv_read + kv_write + B * h * 2 + B * L * keys * 4


def op_bytes(sh: synth.Shape, B: int, op: str, keys: int) -> int:
    """Algorithmic bytes of one launch of a decode-step operation: weights,
    biases and scales once, activations read and written, cache traffic."""
    h, F, V = sh.hidden, sh.ffn, sh.vocab
    wb = 1 if sh.int8 else 2
    if op in ("qkv", "dense", "up", "down"):
        N, K = linear_shapes(sh)[op]
        w = N * K * wb + N * 2 + (N * 2 if sh.int8 else 0)
        act_in = B * K * 2
        act_out = B * N * 8 if op in ("dense", "down") else B * N * 2   # float32 residual r+w
        return w + act_in + act_out
    if op == "attn":
        return B * 2 * keys * h * 2 + B * keys * 4 + 2 * B * h * 2
    if op == "layernorm":
        return B * h * 4 + B * h * 2 + 2 * h * 2
    if op == "embed":
        return B * h * 2 + B * h * 4 + 2 * h * 2 + B * 4
    if op == "head":
        return V * h * 2 + B * h * 2 + B * 4
    raise ValueError(op)


OP_NAMES = {"embed": "embedding gather + LN", "layernorm": "LayerNorm",
            "qkv": "fused QKV + bias + K/V append", "attn": "split-KV ALiBi decode attention",
            "dense": "attention output projection + bias + residual",
            "up": "MLP up + bias + GeLU", "down": "MLP down + bias + residual",
            "head": "tied LM head + argmax"}
KERNEL_SOURCES = {
    "gemv_tc_kernel": ["k_gemv_tc.cu", "tc_ops.cuh", "tile_ops.cuh", "common.cuh", "kernels.h"],
    "linear_kernel": ["k_linear.cu", "tile_ops.cuh", "common.cuh", "kernels.h"],
    "attn_decode_kernel": ["k_attn.cu", "attn_ops.cuh", "common.cuh", "kernels.h"],
    "layernorm_kernel": ["k_norm.cu", "norm_ops.cuh", "common.cuh", "kernels.h"],
    "embed_kernel": ["k_norm.cu", "norm_ops.cuh", "common.cuh", "kernels.h"],
}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def kernel_source_digest(kernel: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(kernel, []):
        with open(os.path.join(ROOT, "bloom_decoder_token_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(op: str, kernel: str, workload: str):
    """dram__bytes_read.sum + dram__bytes_write.sum of one launch of this
    operation's kernel as an ncu capture recorded it for this workload, or None
    when there is none or the kernel's sources changed since."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    d = json.load(open(TRAFFIC_FILE)).get("kernels", {}).get(f"{op}/{kernel}")
    if not d or d.get("kernel_source_sha256") != kernel_source_digest(kernel):
        return None
    return d.get("bytes_per_launch", {}).get(workload)


# ------------------------------------------------------------------ clocks
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(index), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.close()
        rows = [l.split(",") for l in open(self.f.name).read().strip().splitlines() if l.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle
def oracle_sample(sh, w_host, ids, mask, rows, decode_steps):
    """Time the oracle on a bounded sample of the job: the prefill of the first
    `rows` prompts, then `decode_steps` decode steps of those rows.  Returns
    (seconds of the sample, extrapolated seconds of the whole job, threads):
    the oracle's cost is linear in rows, so the job (B rows, one prefill and
    new_tokens - 1 decode steps) takes B / rows * (prefill + (new_tokens - 1)
    * mean decode step)."""
    import oracle
    om = oracle.Model(w_host)
    B, T = ids.shape
    seqs = om.new_seqs(rows, T + decode_steps + 1)
    t0 = time.perf_counter()
    lg = om.prefill(seqs, ids[:rows].numpy(), mask[:rows].numpy())
    t1 = time.perf_counter()
    for _ in range(decode_steps):
        lg = om.decode(seqs, lg.argmax(axis=1).astype("int32"))
    t2 = time.perf_counter()
    step = (t2 - t1) / max(decode_steps, 1)
    job = B / rows * ((t1 - t0) + (sh.new_tokens - 1) * step)
    return t2 - t0, job, oracle.num_threads()


# ------------------------------------------------------------------ distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def maybe_init_dist(world):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group("gloo")


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ reference arm
def run_reference(args, sh):
    """The CPU oracle as it stands, on the host cores: every step is one
    bounded sample of the workload (the prefill of one prompt and
    `ref_decode_steps` decode steps of it), extrapolated to the whole job."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    ids, mask = synth.make_prompts(sh, seed=0)
    w = synth.make_weights(sh, seed=0, device="cpu")
    steps = args.ref_decode_steps
    samples, jobs = [], []
    cores = 0
    for i in range(args.warmup + args.steps):
        dt, job, cores = oracle_sample(sh, w, ids, mask, 1, steps)
        if i >= args.warmup:
            samples.append(dt)
            jobs.append(job)
    B = ids.shape[0]
    job = sum(jobs) / len(jobs)
    value = B * sh.new_tokens / job
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(samples) / len(samples), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,0.02) weights, random prompts)",
        "config": workload_config(sh, B, int(ids.shape[1]), 1),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"per step: prefill of 1 of the {B} prompts + {steps} decode "
                                   f"steps of it, float64 oracle; tokens/s of the whole job "
                                   f"extrapolated linearly in rows and decode steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(sh, B, T, world):
    return {"workload": f"{sh.name}: {sh.n_layer} layers, h {sh.hidden}, {sh.n_head} heads x "
                        f"{sh.head_dim}, MLP {sh.ffn}, vocab {sh.vocab}"
                        f"{', int8 weight-only block linears' if sh.int8 else ''}, batch {B}, "
                        f"prompt {T}{' (left-padded, lengths 8..32)' if sh.ragged else ''}, "
                        f"{sh.new_tokens} greedy tokens",
            "batch": B, "prompt": T, "new_tokens": sh.new_tokens,
            "parallelism": f"replicas x{world}",
            "l2": f"inputs larger than L2: {weight_bytes(sh) / 1e9:.2f} GB of weights streamed "
                  f"per decode step vs {L2_BYTES / 2 ** 20:.0f} MiB L2"}


# ------------------------------------------------------------------ our arm
def model_flags(args, bg):
    return ((bg.FLAG_NO_PDL if args.no_pdl else 0) |
            (bg.FLAG_NO_LN_FUSION if args.no_ln_fusion else 0) |
            (bg.FLAG_NO_TC_GEMM if args.no_tc_gemm else 0))


def time_decode_steps(gm, kv, tok, steps, stream, dev):
    """Mean time of `steps` decode steps (graph replays) with CUDA events."""
    gm.decode_step(kv, tok, tok)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    a.record(stream)
    for _ in range(steps):
        gm.decode_step(kv, tok, tok)
    b.record(stream)
    torch.cuda.synchronize(dev)
    return a.elapsed_time(b) / steps


def decode_series(gm, sh, batches, dev, stream, hbm):
    """Decode step time of the model at several batch sizes: prefill of the
    first B prompts of the workload, then the 99 decode steps of a generation
    (every step reads one more key per sequence), timed as graph replays."""
    out = {}
    ids_all, mask_all = synth.make_prompts(sh.with_(batch=max(batches)), seed=0)
    for B in batches:
        ids, mask = ids_all[:B].to(dev), mask_all[:B].to(dev)
        T = ids.shape[1]
        n_steps = sh.new_tokens - 1
        kv = gm.new_kv(B, T + sh.new_tokens)
        tok = torch.empty(B, dtype=torch.int32, device=dev)
        gm.prefill(kv, ids, mask, out_tokens=tok)
        ms = time_decode_steps(gm, kv, tok, n_steps - 1, stream, dev)   # first step untimed
        keys = T + sh.new_tokens // 2
        nbytes = decode_step_bytes(sh, B, keys)
        gbs = nbytes / (ms / 1e3) / 1e9
        out[str(B)] = {"decode_step_ms": ms, "ms_per_token": ms / B, "tokens_per_s": B / ms * 1e3,
                       "decode_step_bytes": nbytes, "decode_hbm_gbs": gbs,
                       "decode_hbm_frac": gbs / hbm}
        del kv
    return out


def prefill_flops(sh: synth.Shape, B: int, T: int) -> float:
    """Algorithmic FLOPs of one prefill of B full prompts of T tokens: the four
    block linears for every token, causal attention (QK^T and PV over the keys
    each query sees), and the LM head for the last token of each row."""
    h, L = sh.hidden, sh.n_layer
    lin = 2.0 * B * T * sum(N * K for N, K in linear_shapes(sh).values()) * L
    att = 2.0 * 2.0 * B * L * h * (T * (T + 1) / 2.0)
    head = 2.0 * B * sh.vocab * h
    return lin + att + head


def op_gemm_line(shape: str, dev, bg, reps: int = 0):
    """One prefill GEMM (bloom_op_gemm, bias, no activation) of M x N x K at
    bf16, timed with CUDA events over launches alternating between two weight
    copies (together larger than L2 for the shapes of interest), beside
    torch.nn.functional.linear (cuBLAS) on the same operands."""
    M, N, K = (int(v) for v in shape.split("x"))
    g = torch.Generator(device=dev).manual_seed(5)
    x = torch.randn(M, K, device=dev, generator=g).to(torch.bfloat16)
    ws = [(torch.randn(N, K, device=dev, generator=g) * 0.02).to(torch.bfloat16) for _ in range(2)]
    b = torch.zeros(N, device=dev, dtype=torch.bfloat16)
    y = torch.empty(M, N, device=dev, dtype=torch.bfloat16)
    flop = 2.0 * M * N * K
    reps = reps or max(5, min(200, int(2e13 / flop)))
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        for i in range(3):
            fn(i)
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        c = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(reps):
            fn(i)
        c.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(c) / reps

    ms = timed(lambda i: bg.op_gemm(x, ws[i % 2], bias=b, y=y))
    ms_ref = timed(lambda i: torch.nn.functional.linear(x, ws[i % 2], b))
    peak, src = bf16_peak()
    tf = flop / (ms / 1e3) / 1e12
    return {"shape": shape, "ms": ms, "tflops": tf, "peak_tflops": peak, "frac": tf / peak,
            "peak_source": src, "cublas_ms": ms_ref, "cublas_tflops": flop / (ms_ref / 1e3) / 1e12,
            "reps": reps}


def prefill_extra(name, B, T, dev, args, bg):
    """Whole prefill of B prompts of T tokens through bloom_prefill on a preset
    stack (its own model, freed afterwards): time (CUDA events), TFLOP/s and
    the fraction of the dense bf16 peak."""
    sh = synth.PRESETS[name].with_(batch=B, prompt=T, new_tokens=1)
    w = synth.make_weights(sh, seed=0, device=dev)
    gm = bg.Model(w, max_batch=B, max_tokens=B * T, max_seq=T + 1, flags=model_flags(args, bg))
    g = torch.Generator().manual_seed(7)
    ids = torch.randint(0, sh.vocab, (B, T), generator=g, dtype=torch.int64).to(torch.int32).to(dev)
    mask = torch.ones(B, T, dtype=torch.uint8, device=dev)
    kv = gm.new_kv(B, T + 1)
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(2):
        gm.prefill(kv, ids, mask, out_tokens=tok)
    torch.cuda.synchronize(dev)
    times = []
    for _ in range(3):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        gm.prefill(kv, ids, mask, out_tokens=tok)
        b.record(stream)
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b))
    gm.check_device()
    gm.close()
    del gm, w, kv
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    ms = min(times)
    fl = prefill_flops(sh, B, T)
    peak, src = bf16_peak()
    return {"workload": f"{name}: {sh.n_layer} layers, h {sh.hidden}, prefill of {B} x {T} tokens",
            "prefill_ms": ms, "tflop": fl / 1e12, "tflops": fl / (ms / 1e3) / 1e12,
            "bf16_peak_tflops": peak, "peak_source": src,
            "frac_of_bf16_peak": fl / (ms / 1e3) / 1e12 / peak}


def kernel_shares(gm, sh, B, T, dev, reps=3):
    """Each operation's share of one decode step, timed launch by launch with
    CUDA events on the step's stream (bloom_decode_profile: the same kernels
    as a graph replay, each starting after its predecessor has finished), in
    the middle of a generation (cache about half full).  Per (op, kernel):
    launches, total ms (median over `reps` steps), share, algorithmic bytes per
    launch and the bandwidth they imply."""
    ids, mask = synth.make_prompts(sh.with_(batch=B), seed=0)
    kv = gm.new_kv(B, T + sh.new_tokens)
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    gm.prefill(kv, ids.to(dev), mask.to(dev), out_tokens=tok)
    for _ in range(max(0, min(sh.new_tokens // 2 - 1, sh.new_tokens - 1 - reps))):
        gm.decode_step(kv, tok, tok)
    keys = kv.len + 1
    runs = [gm.decode_profile(kv, tok, tok) for _ in range(reps)]
    torch.cuda.synchronize(dev)
    per = {}
    for i, (op, kern, _) in enumerate(runs[0]):
        ms = statistics.median(r[i][2] for r in runs)
        d = per.setdefault((op, kern), {"op": op, "kernel": kern, "launches": 0, "ms": 0.0})
        d["launches"] += 1
        d["ms"] += ms
    total = sum(d["ms"] for d in per.values())
    rows = []
    for d in sorted(per.values(), key=lambda d: -d["ms"]):
        nb = op_bytes(sh, B, d["op"], keys + 1)
        per_launch = d["ms"] / d["launches"]
        rows.append({**d, "share": d["ms"] / total, "ms_per_launch": per_launch,
                     "bytes_per_launch": nb, "gbs": nb / (per_launch / 1e3) / 1e9})
    return rows, total, keys


def sampling_extra(gm, sh, B, T, S, ids_d, mask_d, dev, stream, bg, hbm):
    """Per-member temperature + top-p sampling on the bench workload: the
    sampling kernel alone on B rows of V float32 logits (CUDA events; bytes =
    one read of the logits + the per-row parameters and tokens), and decode
    steps with sampling (logits written, then sampled) against greedy ones."""
    V = sh.vocab
    g = torch.Generator().manual_seed(3)
    temps = (0.5 + torch.rand(B, generator=g)).to(dev)
    tops = torch.full((B,), 0.9).to(dev)
    u = torch.rand(B, generator=g).to(dev)
    lg = torch.empty(B, V, dtype=torch.float32, device=dev)
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    n = min(20, S - T - 1)

    def steps(sampled):
        kv = gm.new_kv(B, S)
        gm.prefill(kv, ids_d, mask_d, out_tokens=tok)
        for _ in range(2):   # warm-up (graph capture)
            if sampled:
                gm.decode_step_sampled(kv, tok, temps, tops, u, lg, out_tokens=tok)
            else:
                gm.decode_step(kv, tok, tok, logits=lg)
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n - 2):
            if sampled:
                gm.decode_step_sampled(kv, tok, temps, tops, u, lg, out_tokens=tok)
            else:
                gm.decode_step(kv, tok, tok, logits=lg)
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / (n - 2)

    greedy_ms = steps(False)
    sampled_ms = steps(True)
    line = op_sample_line(lg, temps, tops, u, dev, stream, bg, hbm)
    line.update({"workload": f"{sh.name}: B {B}, V {V} (the step's logits), temperature 0.5-1.5, "
                             f"top-p 0.9",
                 "decode_step_ms_greedy_with_logits": greedy_ms,
                 "decode_step_ms_sampled": sampled_ms})
    return line


def offload_extra(gm, sh, B, T, S, ids_d, mask_d, dev, stream):
    """Decode steps with the K / V of the upper half of the layers in page-locked
    host memory (read and written by the kernels over the host link) against
    the same steps with the whole cache in HBM.  The KV bytes of the offloaded
    layers over the added time give the bandwidth the host link delivered."""
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    n = min(20, S - T - 1)
    half = sh.n_layer // 2
    res = {}
    for name, off in (("hbm", None), ("offloaded", half)):
        kv = gm.new_kv(B, S, offload_from=off)
        gm.prefill(kv, ids_d, mask_d, out_tokens=tok)
        for _ in range(2):
            gm.decode_step(kv, tok, tok)
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n - 2):
            gm.decode_step(kv, tok, tok)
        b.record(stream)
        torch.cuda.synchronize(dev)
        res[name] = a.elapsed_time(b) / (n - 2)
        del kv
    keys = T + 2 + (n - 2) // 2     # mean keys per step of the timed steps
    kv_bytes = (sh.n_layer - half) * B * 2 * keys * sh.hidden * 2
    extra_ms = res["offloaded"] - res["hbm"]
    return {"workload": f"{sh.name}: B {B}, K / V of layers {half}..{sh.n_layer - 1} in host memory",
            "decode_step_ms_hbm": res["hbm"], "decode_step_ms_offloaded": res["offloaded"],
            "offloaded_kv_bytes_per_step": kv_bytes,
            "host_link_gbs": kv_bytes / (extra_ms / 1e3) / 1e9 if extra_ms > 0 else None}


def op_sample_line(lg, temps, tops, u, dev, stream, bg, hbm, reps: int = 20):
    """The sampling kernel alone on these logits (CUDA events); its bytes are
    one read of the logits plus the per-row parameters and tokens."""
    B, V = lg.shape
    out = torch.empty(B, dtype=torch.int32, device=dev)
    for _ in range(3):
        bg.op_sample(lg, temps, tops, u, out=out)
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        bg.op_sample(lg, temps, tops, u, out=out)
    b.record(stream)
    torch.cuda.synchronize(dev)
    us = a.elapsed_time(b) / reps * 1e3
    nbytes = B * V * 4 + B * 16
    gbs = nbytes / (us / 1e6) / 1e9
    return {"sample_kernel_us": us, "bytes_per_launch": nbytes, "achieved_gbs": gbs,
            "frac_of_hbm": gbs / hbm}


def extra_stack(name, batches, dev, args, bg, hbm):
    """Decode series of another preset (its own model, freed afterwards)."""
    sh = synth.PRESETS[name]
    ids, _ = synth.make_prompts(sh.with_(batch=max(batches)), seed=0)
    T = ids.shape[1]
    w = synth.make_weights(sh, seed=0, device=dev)
    gm = bg.Model(w, max_batch=max(batches), max_tokens=max(batches) * T,
                  max_seq=T + sh.new_tokens, flags=model_flags(args, bg))
    stream = torch.cuda.current_stream(dev)
    out = decode_series(gm, sh, batches, dev, stream, hbm)
    gm.close()
    del gm, w
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return {"workload": workload_config(sh, max(batches), T, 1)["workload"], "by_batch": out}


def run_ours(args, sh):
    import bloom_decoder_token_gb300 as bg

    world, rank, local = dist_env()
    maybe_init_dist(world)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ids, mask = synth.make_prompts(sh, seed=0)
    B, T = ids.shape
    n_new = sh.new_tokens
    S = T + n_new
    series = SERIES_BATCHES if (sh.name == "7b1" and not args.no_extras) else ()
    max_b = max((B,) + tuple(series))
    w = synth.make_weights(sh, seed=0, device=dev)
    gm = bg.Model(w, max_batch=max_b, max_tokens=max_b * T, max_seq=S, flags=model_flags(args, bg))
    kv = gm.new_kv(B, S)
    ids_d, mask_d = ids.to(dev), mask.to(dev)
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def generation():
        gm.prefill(kv, ids_d, mask_d, out_tokens=tok)
        for i in range(1, n_new):
            gm.decode_step(kv, tok, tok)

    for _ in range(args.warmup):
        generation()
    torch.cuda.synchronize(dev)
    clk = Clocks(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        generation()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    ms_total = e0.elapsed_time(e1)
    clocks = clk.stop()
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / args.steps
    tokens_all = sum_over_ranks(args.steps * B * n_new, world)
    value = tokens_all / (ms_total / 1e3)

    # prefill alone, and the decode step as the rest of the generation
    prefill_ms = []
    for _ in range(3):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        gm.prefill(kv, ids_d, mask_d, out_tokens=tok)
        b.record(stream)
        torch.cuda.synchronize(dev)
        prefill_ms.append(a.elapsed_time(b))
    pre_ms = min(prefill_ms)
    dec_ms = (ms_step - pre_ms) / (n_new - 1)
    hbm, src = peaks()
    step_bytes = decode_step_bytes(sh, B, T + n_new // 2)
    dec_gbs = step_bytes / (dec_ms / 1e3) / 1e9

    # per-operation shares of a decode step; the roofline kernel is the largest
    shares, prof_total, prof_keys = kernel_shares(gm, sh, B, T, dev)
    top = shares[0]
    workload_key = f"{sh.name}/B{B}"
    traffic = recorded_traffic(top["op"], top["kernel"], workload_key)

    # end to end through the public API with host buffers
    ids_h = ids.contiguous().pin_memory()
    mask_h = mask.contiguous().pin_memory()
    out_h = torch.empty(n_new, B, dtype=torch.int32).pin_memory()
    kv2 = gm.new_kv(B, S)
    gm.generate(kv2, ids_h, mask_h, n_new, out_h)
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        gm.generate(kv2, ids_h, mask_h, n_new, out_h)
    t1 = time.perf_counter()
    e2e_s = max_over_ranks(t1 - t0, world)
    e2e_value = tokens_all / e2e_s
    del kv2

    launches_prefill = 2 + 7 * sh.n_layer + 2
    launches = args.steps * (launches_prefill + (n_new - 1) * gm.decode_launches(B))

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        wh = w.to("cpu")
        rows, steps = 1, args.cpu_decode_steps
        dt, job, cores = oracle_sample(sh, wh, ids, mask, rows, steps)
        cpu = {"value": B * n_new / job, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"prefill of {rows} of the {B} prompts + {steps} decode steps of it "
                         f"({dt:.1f} s, float64 oracle); tokens/s of the whole job extrapolated "
                         f"linearly in rows and decode steps"}
        del wh

    extras = {}
    if series:
        extras["decode_by_batch"] = decode_series(gm, sh, series, dev, stream, hbm)
        extras["sampling"] = sampling_extra(gm, sh, B, T, S, ids_d, mask_d, dev, stream, bg, hbm)
        extras["kv_offload"] = offload_extra(gm, sh, B, T, S, ids_d, mask_d, dev, stream)
    gm.close()
    del gm, kv
    torch.cuda.synchronize(dev)
    if not args.no_extras and sh.name == "7b1":
        del w
        torch.cuda.empty_cache()
        extras["int8_7b1"] = extra_stack("7b1int8", (1, 8, 32, 128), dev, args, bg, hbm)
        extras["cfg_176b14"] = extra_stack("176b14", (1, 8, 32, 128, 256), dev, args, bg, hbm)
        extras["prefill_176b14_4x2048"] = prefill_extra("176b14", 4, 2048, dev, args, bg)
        extras["prefill_7b1_128x16"] = prefill_extra("7b1", 128, 16, dev, args, bg)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8" if sh.int8 else "bf16",
            "data": "synthetic: seeded N(0,0.02) bf16 weights, biases 0, LN 1/0, random prompts",
            "config": workload_config(sh, B, T, world),
            "ms_per_token": ms_total / (args.steps * B * n_new),
            "decode_step_ms": dec_ms, "prefill_ms": pre_ms,
            "decode_step_bytes": step_bytes,
            "decode_hbm_gbs": dec_gbs,
            "decode_hbm_frac": dec_gbs / hbm,
            "roofline": {"bound": "hbm", "kernel": f"{top['kernel']} ({OP_NAMES[top['op']]})",
                         "achieved": top["gbs"], "peak": hbm, "unit": "GB/s",
                         "frac": top["gbs"] / hbm, "traffic": traffic, "peak_source": src,
                         "bytes_per_launch": top["bytes_per_launch"],
                         "launch_ms": top["ms_per_launch"], "step_share": top["share"],
                         "timing": "CUDA events on the decode stream, one event per launch, "
                                   "launches serialised (bloom_decode_profile)"},
            "kernel_shares": {"workload": workload_key, "keys": prof_keys,
                              "serialised_step_ms": prof_total,
                              "rows": [{k: r[k] for k in ("op", "kernel", "launches", "ms",
                                                          "share", "ms_per_launch",
                                                          "bytes_per_launch", "gbs")}
                                       for r in shares]},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT,
                    "h2d_bytes_per_step": B * T * 5, "d2h_bytes_per_step": n_new * B * 4},
            "gpu_launches": launches,
            "clocks": clocks,
            **extras,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(synth.PRESETS))
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--new-tokens", type=int, default=None)
    ap.add_argument("--layers", type=int, default=None, help="decoder layers (default: the preset's)")
    ap.add_argument("--prompt", type=int, default=None, help="padded prompt length (default: the preset's)")
    ap.add_argument("--cpu-decode-steps", type=int, default=4)
    ap.add_argument("--ref-decode-steps", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill-only", default=None, metavar="PRESET:BxT",
                    help="only time one whole prefill, e.g. 176b14:4x2048, and print its line")
    ap.add_argument("--op-gemm", default=None, metavar="MxNxK",
                    help="only time one prefill GEMM of this shape (and cuBLAS beside it)")
    ap.add_argument("--op-reps", type=int, default=0, help="launches timed by --op-gemm (0: by size)")
    ap.add_argument("--op-sample", default=None, metavar="BxV",
                    help="only time the sampling kernel on B rows of V seeded logits "
                         "(N(0, 2), temperature 0.5-1.5, top-p 0.9)")
    ap.add_argument("--no-extras", action="store_true",
                    help="only the workload itself (no batch series, int8 or 176B-shape keys)")
    ap.add_argument("--no-pdl", action="store_true", help="launch without programmatic dependent launch")
    ap.add_argument("--no-ln-fusion", action="store_true", help="separate LayerNorm kernels")
    ap.add_argument("--no-tc-gemm", action="store_true",
                    help="every linear on the weight-streaming kernel instead of tcgen05")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    sh = synth.PRESETS[args.config]
    batch = args.batch or DEFAULT_BATCH.get(args.config)
    if batch:
        sh = sh.with_(batch=batch)
    if args.new_tokens:
        sh = sh.with_(new_tokens=args.new_tokens)
    if args.layers:
        sh = sh.with_(n_layer=args.layers)
    if args.prompt:
        sh = sh.with_(prompt=args.prompt)
    if args.impl == "reference":
        run_reference(args, sh)
    elif args.op_gemm:
        import bloom_decoder_token_gb300 as bg
        torch.cuda.set_device(0)
        print(json.dumps({"op_gemm": op_gemm_line(args.op_gemm, torch.device("cuda", 0), bg,
                                                  args.op_reps)}), flush=True)
    elif args.op_sample:
        import bloom_decoder_token_gb300 as bg
        torch.cuda.set_device(0)
        dev = torch.device("cuda", 0)
        B, V = (int(v) for v in args.op_sample.split("x"))
        g = torch.Generator().manual_seed(3)
        lg = (torch.randn(B, V, generator=g) * 2.0).to(dev)
        temps = (0.5 + torch.rand(B, generator=g)).to(dev)
        tops = torch.full((B,), 0.9).to(dev)
        u = torch.rand(B, generator=g).to(dev)
        hbm, _ = peaks()
        line = op_sample_line(lg, temps, tops, u, dev, torch.cuda.current_stream(dev), bg, hbm)
        line["shape"] = args.op_sample
        print(json.dumps({"op_sample": line}), flush=True)
    elif args.prefill_only:
        import bloom_decoder_token_gb300 as bg
        name, bt = args.prefill_only.split(":")
        B, T = (int(v) for v in bt.split("x"))
        torch.cuda.set_device(0)
        print(json.dumps({"prefill_only": prefill_extra(name, B, T, torch.device("cuda", 0), args,
                                                        bg)}), flush=True)
    else:
        run_ours(args, sh)


if __name__ == "__main__":
    main()
