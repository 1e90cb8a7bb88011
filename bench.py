"""Benchmark: greedy KV-cached generation through a BLOOM decoder stack on GB300.

One step = one whole generation of the workload: prefill of the B padded
prompts, then new_tokens - 1 decode steps (graph replays), argmax fed back on
the device.  value = tokens/s = B * new_tokens / (time per step), the pages'
per-token cost being its inverse (wall time / (batch x tokens)).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config 560m|7b1|7b1int8|176b14|block] [--batch B]

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


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------------ byte model
def weight_bytes(sh: synth.Shape) -> int:
    """Algorithmic bytes of all weights one decode step reads once."""
    h, F, V, L = sh.hidden, sh.ffn, sh.vocab, sh.n_layer
    per = 0
    for N, K in [(3 * h, h), (h, h), (F, h), (h, F)]:
        per += N * K * (1 if sh.int8 else 2) + N * 2 + (N * 2 if sh.int8 else 0)   # W, bias, scales
    per += 4 * h * 2                                                               # 2 LayerNorms
    return L * per + V * h * 2 + 4 * h * 2                                         # + head E, ln_f, emb LN


def decode_step_bytes(sh: synth.Shape, B: int, keys: int) -> int:
    """Weights + KV read (keys slots, incl. the new one) + KV write + embedding rows."""
    h, L = sh.hidden, sh.n_layer
    kv_read = B * L * 2 * keys * h * 2
    kv_write = B * L * 2 * h * 2
    return weight_bytes(sh) + kv_read + kv_write + B * h * 2 + B * L * keys * 4


def head_launch_bytes(sh: synth.Shape, B: int) -> int:
    return sh.vocab * sh.hidden * 2 + B * sh.hidden * 2 + B * 4


# ------------------------------------------------------------------ measured DRAM traffic
# The LM head + argmax runs on the tensor-core decode kernel from 8 sequences
# on (unless disabled), else on the weight-streaming kernel.
HEAD_KERNELS = {
    "gemv_tc": ("gemv_tc_kernel (tensor-core LM head + argmax)",
                ["k_gemv_tc.cu", "tc_ops.cuh", "tile_ops.cuh", "common.cuh", "kernels.h"]),
    "linear": ("linear_kernel (weight-streaming LM head + argmax)",
               ["k_linear.cu", "tile_ops.cuh", "common.cuh", "kernels.h"]),
}
TC_HEAD_MIN_B = 8
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "lm_head_traffic.json")


def head_kernel(B: int, tc: bool) -> str:
    return "gemv_tc" if tc and B >= TC_HEAD_MIN_B else "linear"


def head_source_digest(kernel: str) -> str:
    h = hashlib.sha256()
    for f in HEAD_KERNELS[kernel][1]:
        with open(os.path.join(ROOT, "bloom_decoder_token_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def head_traffic(sh: synth.Shape, B: int, kernel: str):
    """dram__bytes_read.sum + dram__bytes_write.sum of one LM-head launch as an
    ncu capture recorded it for this workload and kernel, or None when there is
    no capture for it or the kernel's sources changed since."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    d = json.load(open(TRAFFIC_FILE)).get("kernels", {}).get(kernel)
    if not d or d.get("kernel_source_sha256") != head_source_digest(kernel):
        return None
    return d.get("bytes_per_launch", {}).get(f"{sh.name}/B{B}")


def measure_head(gm, sh, B, dev, stream, reps=50):
    """Dominant kernel: the tied LM head + argmax (largest single weight stream),
    timed alone with CUDA events on its stream."""
    xn = torch.randn(B, sh.hidden, device=dev).to(torch.bfloat16)
    ht = torch.empty(B, dtype=torch.int32, device=dev)
    for _ in range(3):
        gm.lm_head(xn, ht)
    torch.cuda.synchronize(dev)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        gm.lm_head(xn, ht)
    b.record(stream)
    torch.cuda.synchronize(dev)
    head_ms = a.elapsed_time(b) / reps
    head_bytes = head_launch_bytes(sh, B)
    return head_ms, head_bytes, head_bytes / (head_ms / 1e3) / 1e9


def run_roofline_only(args, sh):
    """Only the dominant kernel's measurement (the command an ncu capture of its
    DRAM counters runs)."""
    import bloom_decoder_token_gb300 as bg
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    B = sh.batch
    w = synth.make_weights(sh.with_(n_layer=1), seed=0, device=dev)
    gm = bg.Model(w, max_batch=B, max_tokens=B * sh.prompt, max_seq=sh.max_seq,
                  flags=bg.FLAG_NO_TC_GEMM if args.no_tc_gemm else 0)
    kernel = head_kernel(B, not args.no_tc_gemm)
    head_ms, head_bytes, head_gbs = measure_head(gm, sh, B, dev, torch.cuda.current_stream(dev))
    hbm, src = peaks()
    print(json.dumps({"roofline_only": True, "workload": f"{sh.name}/B{B}", "kernel": kernel,
                      "launch_ms": head_ms, "bytes_per_launch": head_bytes,
                      "achieved_gbs": head_gbs, "frac": head_gbs / hbm, "peak_source": src,
                      "kernel_source_sha256": head_source_digest(kernel)}), flush=True)
    gm.close()


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
def oracle_sample(sh, w_host, ids, mask, decode_steps):
    """Time the oracle on a bounded sample: prefill + `decode_steps` steps."""
    import oracle
    om = oracle.Model(w_host)
    B, T = ids.shape
    seqs = om.new_seqs(B, T + decode_steps + 1)
    t0 = time.perf_counter()
    lg = om.prefill(seqs, ids.numpy(), mask.numpy())
    for _ in range(decode_steps):
        lg = om.decode(seqs, lg.argmax(axis=1).astype("int32"))
    dt = time.perf_counter() - t0
    return dt, B * (1 + decode_steps), oracle.num_threads()


def host_weights(w):
    return w.to("cpu")


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
    world, rank, _ = dist_env()
    if rank != 0:
        return
    ids, mask = synth.make_prompts(sh, seed=0)
    w = synth.make_weights(sh, seed=0, device="cpu")
    steps = args.ref_decode_steps
    times = []
    for i in range(args.warmup + args.steps):
        dt, ntok, cores = oracle_sample(sh, w, ids, mask, steps)
        if i >= args.warmup:
            times.append(dt)
    per = sum(times) / len(times)
    B = ids.shape[0]
    value = B * (1 + steps) / per
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,0.02) weights, "
        "random prompts)",
        "config": {"workload": sh.name, "batch": B, "prompt": int(ids.shape[1]),
                   "tokens_per_step": 1 + steps},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"prefill + {steps} decode steps of the {sh.name} workload "
                                   f"(B={B}) per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm
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
    w = synth.make_weights(sh, seed=0, device=dev)
    gm = bg.Model(w, max_batch=B, max_tokens=B * T, max_seq=S,
                  flags=(bg.FLAG_NO_PDL if args.no_pdl else 0) |
                  (bg.FLAG_NO_LN_FUSION if args.no_ln_fusion else 0) |
                  (bg.FLAG_PERSISTENT if args.persistent else 0) |
                  (bg.FLAG_NO_TC_GEMM if args.no_tc_gemm else 0))
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

    # decode step alone: mean over the generation's 99 steps (graph replays)
    prefill_ms = []
    for _ in range(3):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        gm.prefill(kv, ids_d, mask_d, out_tokens=tok)
        b.record(stream)
        torch.cuda.synchronize(dev)
        prefill_ms.append(a.elapsed_time(b))
        for i in range(1, n_new):
            gm.decode_step(kv, tok, tok)
    torch.cuda.synchronize(dev)
    pre_ms = min(prefill_ms)
    dec_ms = (ms_step - pre_ms) / (n_new - 1)
    mean_keys = T + n_new / 2.0
    step_bytes = decode_step_bytes(sh, B, int(round(mean_keys)))
    hbm, src = peaks()
    dec_gbs = step_bytes / (dec_ms / 1e3) / 1e9

    head_ms, head_bytes, head_gbs = measure_head(gm, sh, B, dev, stream)
    kernel = head_kernel(B, not args.no_tc_gemm)
    traffic = args.head_traffic if args.head_traffic is not None else head_traffic(sh, B, kernel)

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

    launches_prefill = 2 + 7 * sh.n_layer + 2
    launches = args.steps * (launches_prefill + (n_new - 1) * gm.decode_launches(B))

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        wh = host_weights(w)
        steps = args.cpu_decode_steps
        dt, ntok, cores = oracle_sample(sh, wh, ids, mask, steps)
        cpu = {"value": ntok / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"prefill + {steps} decode steps of the same workload (B={B}), "
                         f"{dt:.1f} s, fp64"}
        del wh

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8" if sh.int8 else "bf16",
            "data": "synthetic: seeded N(0,0.02) bf16 weights, biases 0, LN 1/0, random prompts",
            "config": {"workload": f"{sh.name}: {sh.n_layer} layers, h {sh.hidden}, "
                                   f"{sh.n_head} heads, vocab {sh.vocab}, batch {B}, prompt {T}"
                                   f"{' (left-padded, lengths 8..32)' if sh.ragged else ''}, "
                                   f"{n_new} greedy tokens",
                       "batch": B, "prompt": T, "new_tokens": n_new,
                       "parallelism": f"replicas x{world}",
                       "l2": f"inputs larger than L2: {weight_bytes(sh) / 1e9:.2f} GB of "
                             f"weights streamed per decode step vs {L2_BYTES / 2**20:.0f} MiB L2"},
            "ms_per_token": ms_total / (args.steps * B * n_new),
            "decode_step_ms": dec_ms, "prefill_ms": pre_ms,
            "decode_step_bytes": step_bytes,
            "decode_hbm_gbs": dec_gbs,
            "decode_hbm_frac": dec_gbs / hbm,
            "roofline": {"bound": "hbm", "kernel": HEAD_KERNELS[kernel][0],
                         "achieved": head_gbs, "peak": hbm, "unit": "GB/s",
                         "frac": head_gbs / hbm, "traffic": traffic,
                         "peak_source": src, "bytes_per_launch": head_bytes,
                         "launch_ms": head_ms},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT,
                    "h2d_bytes_per_step": B * T * 5, "d2h_bytes_per_step": n_new * B * 4},
            "gpu_launches": launches,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    gm.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="560m", choices=sorted(synth.PRESETS))
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--new-tokens", type=int, default=None)
    ap.add_argument("--layers", type=int, default=None, help="decoder layers (default: the preset's)")
    ap.add_argument("--prompt", type=int, default=None, help="padded prompt length (default: the preset's)")
    ap.add_argument("--cpu-decode-steps", type=int, default=8)
    ap.add_argument("--ref-decode-steps", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-pdl", action="store_true", help="launch without programmatic dependent launch")
    ap.add_argument("--no-ln-fusion", action="store_true", help="separate LayerNorm kernels")
    ap.add_argument("--persistent", action="store_true",
                    help="decode steps as one persistent cooperative launch (batches <= 16)")
    ap.add_argument("--no-tc-gemm", action="store_true",
                    help="prefill linears on the weight-streaming kernel instead of tcgen05")
    ap.add_argument("--head-traffic", type=float, default=None,
                    help="dram bytes per LM-head launch from an ncu capture of this kernel "
                         "(default: the recorded capture, if the kernel is unchanged)")
    ap.add_argument("--roofline-only", action="store_true",
                    help="only time the dominant kernel (LM head + argmax) and print its line")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    sh = synth.PRESETS[args.config]
    if args.batch:
        sh = sh.with_(batch=args.batch)
    if args.new_tokens:
        sh = sh.with_(new_tokens=args.new_tokens)
    if args.layers:
        sh = sh.with_(n_layer=args.layers)
    if args.prompt:
        sh = sh.with_(prompt=args.prompt)
    if args.impl == "reference":
        run_reference(args, sh)
    elif args.roofline_only:
        run_roofline_only(args, sh)
    else:
        run_ours(args, sh)


if __name__ == "__main__":
    main()
