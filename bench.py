"""Batch-1 decode benchmark of the persistent megakernel on GB300.

Default workload: the Qwen3-0.6B-shaped decoder (28 layers, hidden 1024, 16/8
heads, head_dim 128, MLP 3072, tied 151936 vocab), a 32-token random prompt
and 512 greedy steps, seeded random-init bf16 weights.  One bench step =
reset the KV cache, prefill the prompt (untimed, same kernel, one token per
forward), then ONE persistent launch that runs the 512 greedy forwards; the
CUDA events bracket that launch.  The weights (1.19 GB per forward) exceed
the 129 MB L2, so no L2 flush is needed between steps.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the same workload instead.  Under torchrun every rank decodes its own replica
on its own GPU (independent sessions, no collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "persistent_transformer_megakernel_gb300", "csrc")
PROFILES = os.path.join(ROOT, "profiles")


# the files the decode kernel and its launch are built from; the prefill and
# embedding kernels do not change what the decode kernel reads or writes
DECODE_SOURCES = ("mk_device.cuh", "mk_host.cu", "mk_kernels_d128.cu", "mk_kernels_d64.cu", "mk_kernels_hidden1024.cu",
                  "mk_kernels_hidden2048.cu", "mk_launch.h", "mk_params.h", "mk_plans.h", "ptx.cuh")


def code_only(text):
    """C/C++ source without comments and with whitespace runs collapsed (string
    and character literals kept), so that editing a comment does not count as
    changing the kernel."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_sources_sha256(read=None):
    """Hash of the code (comments excluded) of the decode kernel's sources;
    ``read(name)`` returns a file's text (default: the tree's csrc/)."""
    import hashlib
    if read is None:
        def read(name):
            with open(os.path.join(CSRC, name)) as f:
                return f.read()
    h = hashlib.sha256()
    for name in sorted(DECODE_SOURCES):
        h.update(name.encode())
        h.update(code_only(read(name)).encode())
    return h.hexdigest()


def measured_traffic(workload, forwards_per_launch):
    """DRAM bytes (read + write) per launch from the ncu record of this
    workload, scaled by forwards; None when there is no record or the decode
    kernel's sources changed since it was taken."""
    path = os.path.join(PROFILES, "traffic_%s.json" % workload)
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_sources_sha256") != kernel_sources_sha256():
        return None
    per_fwd = (rec["dram_bytes_read"] + rec["dram_bytes_write"]) / rec["captured_forwards"]
    return per_fwd * forwards_per_launch


def workload_desc(name):
    wl = W.WORKLOADS[name]
    s = W.shape(wl["shape"])
    d = ("%s: %d layers, hidden %d, %d/%d heads, head_dim %d, MLP %d, vocab %d %s%s; "
         "prompt %d + %d greedy steps" % (
             name, s["n_layers"], s["hidden"], s["n_q_heads"], s["n_kv_heads"], s["head_dim"],
             s["intermediate"], s["vocab"], "tied" if s["tied"] else "untied",
             ", MRoPE %s" % (s["mrope_sections"],) if s["mrope_sections"] else "",
             wl["prompt"], wl["steps"]))
    return wl, s, d


def algorithmic_bytes(s, weight_bytes, positions):
    """Bytes one forward must move at slot P: all weights once, the KV cache
    read for positions 0..P and the new K/V row written."""
    kv_row = 2 * s["n_layers"] * s["n_kv_heads"] * s["head_dim"] * 2     # K and V, bf16
    return sum(weight_bytes + kv_row * (P + 1) + kv_row for P in positions)


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", "mk_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
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
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle timing (the reported baseline / the reference arm)
# ---------------------------------------------------------------------------
def cpu_oracle_rate(workload: str, n_forwards: int, threads: int, warmup: int = 0, steps: int = 1):
    """Time the oracle in a child process with a fixed BLAS thread count, at
    the contexts the GPU times: the workload's prompt is laid into the cache
    by the oracle's all-positions path (untimed), then ``warmup`` untimed and
    ``steps`` timed samples of ``n_forwards`` teacher-forced forwards follow
    it.  Returns (seconds per timed sample, first and last context timed)."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(threads)
    code = (
        "import sys,time,json; sys.path.insert(0, %r)\n"
        "import numpy as np, workloads as W, oracle as O\n"
        "wl=W.WORKLOADS[%r]; s=W.shape(wl['shape']); w=W.make_weights(s, seed=0)\n"
        "shp=O.DecoderShape.from_dict(s); Wt=O.decoder.Weights(shp, w); del w\n"
        "n=%d; reps=%d+%d; P0=max(1, wl['prompt'])\n"
        "dec=O.Decoder(shp, None, max_seq=P0+n*reps+2, weights=Wt)\n"
        "p=W.make_prompt(s['vocab_in'], P0+n*reps, seed=1)\n"
        "_, _, K, V = O.prefix_forward(shp, None, p[:P0], logits_for=[P0-1], weights=Wt)\n"
        "dec.K[:, :, :P0]=K; dec.V[:, :, :P0]=V; dec.pos=P0; del K, V\n"
        "out=[]\n"
        "for r in range(reps):\n"
        "    t=time.perf_counter(); dec.generate(p[P0+r*n:P0+(r+1)*n], 0); out.append(time.perf_counter()-t)\n"
        "first=P0+%d*n+1\n"
        "print(json.dumps([out[%d:], first, P0+n*reps]))\n" % (ROOT, workload, n_forwards, warmup, steps,
                                                               warmup, warmup))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("oracle timing failed: " + r.stderr[-2000:])
    dts, c0, c1 = json.loads(r.stdout.strip().splitlines()[-1])
    return dts, (c0, c1)


def reduce_timing(total_ms, units_per_rank, world, device="cpu"):
    """Whole-job throughput of `world` independent replicas: the slowest
    rank's time (all-reduce MAX over the process group) against the units all
    ranks processed.  Returns (max_ms, units per second)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    return total_ms, units_per_rank * world / (total_ms / 1e3)


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# the arms
# ---------------------------------------------------------------------------
def run_reference(args, rank, world):
    """The oracle as it stands, timed on the host cores on bounded samples of
    the same workload: each step is ``--cpu-forwards`` teacher-forced forwards."""
    wl, s, desc = workload_desc(args.workload)
    if rank != 0:
        return
    threads = cpu_threads()
    n = max(1, args.cpu_forwards)
    dts, ctx = cpu_oracle_rate(args.workload, n, threads, warmup=1, steps=args.steps)
    total = sum(dts)
    value = n * len(dts) / total
    line = {
        "impl": "reference", "metric": "batch-1 decode tok/s", "value": value, "unit": "tok/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / len(dts) * 1e3, "us_per_token": total / (n * len(dts)) * 1e6,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded random-init weights, random prompt ids)",
        "config": {"workload": desc},
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": threads, "kind": "oracle",
                         "sample": "%d teacher-forced forwards per step at contexts %d..%d (after the "
                                   "workload's prompt), float64 numpy oracle, BLAS threads %d"
                                   % (n, ctx[0], ctx[1], threads)},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def talker_ttfc(dev, n_prompt=32, chunk=16, reps=4):
    """Time to first chunk on the talker workload (28 layers, hidden 1024,
    3072-entry untied head, MRoPE): host code ids in -> the prompt's 17-way
    input sums (mk_embed_sum) -> the prompt through mk_prefill (sentinel rows,
    three distinct MRoPE position streams) -> greedy forwards streamed through
    the host-mapped mailbox.  Host wall clock from the host ids to the first
    generated id and to the first ``chunk`` ids on the host; best of the reps
    after the first (which allocates the prefill scratch and captures it)."""
    import torch
    import persistent_transformer_megakernel_gb300 as mk
    s = W.shape("tts_talker")
    w = W.make_weights(s, seed=0)
    dec = mk.Decoder(s, w, max_seq=n_prompt + chunk + 8, device=dev)
    del w
    tables = W.make_tts_tables(s["hidden"], seed=3)
    books = torch.from_numpy(tables["codebooks"].view(np.int16)).view(torch.bfloat16).to(dev)
    txt = torch.from_numpy(tables["text"].view(np.int16)).view(torch.bfloat16).to(dev)
    del tables
    codes, text = W.make_tts_codes(n_prompt, seed=2)
    h_codes = torch.as_tensor(codes, dtype=torch.int32).pin_memory()
    h_text = torch.as_tensor(text, dtype=torch.int32).pin_memory()
    h_pos3 = torch.as_tensor(W.make_pos3(0, n_prompt, distinct=True), dtype=torch.int32).pin_memory()
    sid = torch.as_tensor(W.sentinel_ids(n_prompt), dtype=torch.int32).pin_memory()
    first, first_chunk = [], []
    for _ in range(reps):
        dec.reset()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        c_d = h_codes.to(dev, non_blocking=True)
        t_d = h_text.to(dev, non_blocking=True)
        E = mk.embed_sum(books, txt, c_d, t_d)
        dec.prefill(sid.to(dev, non_blocking=True), all_ids=False, embeds=E,
                    pos3=h_pos3.to(dev, non_blocking=True))
        t_first = t_chunk = None
        for i, _tok, _t in dec.decode_stream(None, chunk):
            now = time.perf_counter() - t0
            if t_first is None:
                t_first = now
            if i == chunk - 1:
                t_chunk = now
        first.append(t_first * 1e3)
        first_chunk.append(t_chunk * 1e3)
    dec.close()
    return {"ttfc_talker_ms": min(first_chunk[1:]), "first_id_talker_ms": min(first[1:]),
            "chunk_ids": chunk, "prompt_rows": n_prompt,
            "talker_note": "talker shape (0.6B dims, 3072-entry head, MRoPE 24/20/20): host code ids -> mk_embed_sum -> "
                    "mk_prefill of %d sentinel rows -> MK_DECODE_STREAM greedy forwards; host wall clock to the "
                    "first id and to the first %d ids in the mailbox, best of %d after a first call"
                    % (n_prompt, chunk, reps - 1)}


def run_gpu(args, rank, world):
    import torch
    import persistent_transformer_megakernel_gb300 as mk

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl, s, desc = workload_desc(args.workload)
    n_prompt, n_steps = wl["prompt"], wl["steps"]
    sentinel = wl.get("sentinel", False)

    # CPU baseline before any heavy GPU work (rank 0 at N=1 only): the oracle at
    # one thread and at every host thread, over forwards at the timed contexts
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        threads = cpu_threads()
        n_cpu = max(1, args.cpu_forwards)
        dts, ctx = cpu_oracle_rate(args.workload, n_cpu, threads, warmup=0, steps=1)
        dts1, _ = cpu_oracle_rate(args.workload, n_cpu, 1, warmup=0, steps=1)
        rate = n_cpu / dts[0]
        cpu = {"value": rate, "unit": "tok/s", "cores": threads, "kind": "oracle",
               "single_thread": {"value": n_cpu / dts1[0], "unit": "tok/s", "cores": 1},
               "sample": "%d teacher-forced forwards of the same model at contexts %d..%d (after the "
                         "workload's prompt, laid in by the oracle's all-positions path), float64 numpy "
                         "oracle; value at %d BLAS threads, single_thread at 1" % (n_cpu, ctx[0], ctx[1], threads)}

    w = W.make_weights(s, seed=0)
    max_seq = n_prompt + n_steps + 8
    dec = mk.Decoder(s, w, max_seq=max_seq, device=dev)
    del w
    info = dec.info()
    embeds = pos3 = None
    if sentinel:
        tables = W.make_tts_tables(s["hidden"], seed=3)
        codes, text = W.make_tts_codes(n_prompt, seed=2)
        books = torch.from_numpy(tables["codebooks"].view(np.int16)).view(torch.bfloat16).to(dev)
        txt = torch.from_numpy(tables["text"].view(np.int16)).view(torch.bfloat16).to(dev)
        embeds = mk.embed_sum(books, txt, torch.as_tensor(codes).to(dev), torch.as_tensor(text).to(dev))
        del books, txt, tables
        prompt = W.sentinel_ids(n_prompt)
        pos3 = torch.as_tensor(W.make_pos3(0, n_prompt, distinct=True), device=dev)
    else:
        prompt = W.make_prompt(s["vocab_in"], n_prompt, seed=1)
    d_prompt = torch.as_tensor(prompt, device=dev)
    out = torch.empty(max_seq, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    # the timed unit: greedy steps after the prompt; the talker workload times
    # its sentinel forwards themselves (teacher-forced, no greedy tail)
    if sentinel:
        timed_positions = range(0, n_prompt)

        def prep():
            dec.reset()

        def timed():
            dec.decode(d_prompt, 0, out=out, embeds=embeds, pos3=pos3)
        n_timed = n_prompt
    else:
        timed_positions = range(n_prompt, n_prompt + n_steps)

        def prep():
            dec.reset()
            dec.decode(d_prompt, 0, out=out)

        def timed():
            dec.decode(None, n_steps, out=out)
        n_timed = n_steps

    for _ in range(args.warmup):
        prep()
        timed()
    torch.cuda.synchronize()
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    sampler = ClockSampler(local)
    sampler.start()
    total_ms = 0.0
    for _ in range(args.steps):
        prep()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        timed()
        e1.record(stream)
        e1.synchronize()
        total_ms += e0.elapsed_time(e1)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    total_ms, value = reduce_timing(total_ms, n_timed * args.steps, world, dev)
    if world > 1:
        dist.barrier()
    per_launch_ms = total_ms / args.steps
    bytes_launch = algorithmic_bytes(s, info["weight_bytes"], timed_positions)
    peak, peak_src = load_peaks()
    achieved = bytes_launch / (per_launch_ms / 1e3) / 1e9

    # end to end through the C ABI with host id buffers (copies inside the region)
    e2e_ms = 0.0
    h_prompt = np.asarray(prompt, dtype=np.int32)
    for i in range(args.steps + 1):
        dec.reset()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        if sentinel:
            dec.decode_host(h_prompt, 0, embeds=embeds, pos3=pos3)
        else:
            dec.decode_host(h_prompt, n_steps)
        dt = (time.perf_counter() - t0) * 1e3
        if i > 0:
            e2e_ms += dt
    e2e_tokens = (n_prompt + (0 if sentinel else n_steps)) * args.steps * world
    e2e = {"value": e2e_tokens / (e2e_ms / 1e3), "unit": "tok/s",
           "h2d_bytes_per_step": int(h_prompt.nbytes),
           "d2h_bytes_per_step": int(4 * (n_prompt + (0 if sentinel else n_steps))),
           "note": "mk_decode_host: prompt ids host->device, prompt + greedy forwards in one "
                   "launch, all ids device->host; host wall clock"}

    # streaming: the greedy ids reach a host-mapped mailbox while the launch
    # runs; first-id latency = enqueue to the host seeing the first greedy id
    streaming = None
    if not sentinel and not args.no_ablation:
        dec.reset()
        dec.decode(d_prompt, 0, out=out)
        torch.cuda.synchronize()
        n_st = min(64, n_timed)
        got = list(dec.decode_stream(None, n_st))
        # time to first token from a cold context: host prompt ids in, the
        # prompt consumed one token per forward, the first generated id read
        # from the mailbox (host wall clock)
        dec.reset()
        torch.cuda.synchronize()
        host_prompt = [int(t) for t in prompt]
        first = None
        for i, tok, t in dec.decode_stream(host_prompt, 1):
            if i == len(host_prompt) - 1:
                first = t
        # the same with the batched prefill (tensor-core GEMMs for the prompt):
        # host ids in, prefill, the first generated id back on the host
        pf_ms = []
        for rep in range(4):
            dec.reset()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            first_id = int(dec.prefill(host_prompt)[-1].item())
            pf_ms.append((time.perf_counter() - t0) * 1e3)
        del first_id
        if len(got) == n_st:
            streaming = {"first_id_ms": got[0][2] * 1e3, "last_id_ms": got[-1][2] * 1e3, "ids": n_st,
                         "ttft_ms": None if first is None else first * 1e3,
                         "ttft_prefill_ms": min(pf_ms[1:]),
                         "ttft_prompt": len(host_prompt),
                         "note": "host wall clock from mk_decode_start to the id appearing in the "
                                 "host-mapped mailbox (MK_DECODE_STREAM); first_id/last_id: greedy forwards "
                                 "after a resident prompt; ttft: a %d-token host prompt consumed one token per "
                                 "forward in the same launch, to the first generated id; ttft_prefill: the "
                                 "same prompt through mk_prefill (batched tensor-core GEMMs), best of 3 after "
                                 "a first call that allocates the scratch" % len(host_prompt)}

    if streaming is not None:
        streaming.update(talker_ttfc(dev))

    # launch-overhead ablation: the same phases as one ordinary launch each,
    # i.e. this megakernel relaunched once per phase (its prologue repeats
    # every launch), not a path of separate slim per-op kernels
    ablation = None
    if not args.no_ablation:
        n_ab = min(args.ablation_forwards, n_timed)
        dec.reset()
        if not sentinel:
            dec.decode(d_prompt, 0, out=out)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if sentinel:
            dec.decode(d_prompt[:n_ab], 0, out=out, embeds=embeds, pos3=pos3[:, :n_ab].contiguous(),
                       per_op=True)
        else:
            dec.decode(None, n_ab, out=out, per_op=True)
        e1.record(stream)
        e1.synchronize()
        ab_ms = e0.elapsed_time(e1)
        # the same launches replayed from a captured graph of one forward; a
        # first (untimed) call captures and instantiates it
        g_ms = None
        for timed in (False, True):
            dec.reset()
            if not sentinel:
                dec.decode(d_prompt, 0, out=out)
            torch.cuda.synchronize()
            e0.record(stream)
            if sentinel:
                dec.decode(d_prompt[:n_ab], 0, out=out, embeds=embeds, pos3=pos3[:, :n_ab].contiguous(),
                           per_op="graph")
            else:
                dec.decode(None, n_ab, out=out, per_op="graph")
            e1.record(stream)
            e1.synchronize()
            if timed:
                g_ms = e0.elapsed_time(e1)
        ablation = {"us_per_token": ab_ms * 1e3 / n_ab, "forwards": n_ab,
                    "what": "the persistent kernel's phases, one ordinary launch per phase (the megakernel "
                            "relaunched with one phase each), then the same launches replayed from a graph",
                    "launches_per_forward": 5 * s["n_layers"] + 1,
                    "graph_replay_us_per_token": g_ms * 1e3 / n_ab,
                    "persistent_us_per_token": total_ms * 1e3 / (n_timed * args.steps)}

    if rank != 0:
        return
    line = {
        "metric": "batch-1 decode tok/s",
        "value": value,
        "unit": "tok/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": per_launch_ms,
        "us_per_token": total_ms * 1e3 / (n_timed * args.steps),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 weights / f32 compute",
        "data": "synthetic (seeded random-init weights, random prompt ids)",
        "config": {"workload": desc, "timed": "%d forwards per step in one persistent launch" % n_timed,
                   "l2": "inputs larger than L2: %.2f GB of weights per forward" % (info["weight_bytes"] / 1e9),
                   "grid": info["grid"], "threads": info["threads"],
                   "ring": "%d x %d KB" % (info["stages"], info["stage_bytes"] // 1024),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": measured_traffic(args.workload, n_timed),
                     "peak_source": "%s hbm_gbs (copy bandwidth)" % peak_src,
                     "algorithmic_bytes_per_launch": bytes_launch,
                     "kernel": "mk::mk_decode_kernel<%d, %s>" % (
                         s["head_dim"], {1: "PlanHidden1024", 2: "PlanHidden2048"}.get(info.get("plan", 0), "PlanGeneral"))},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "e2e": e2e,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if ablation is not None:
        line["per_op_ablation"] = ablation
    if streaming is not None:
        line["streaming"] = streaming
    print(json.dumps(line), flush=True)


def ncu_case(args):
    """The small case the ncu captures use: one 16-token prompt launch, then
    one launch of 8 greedy forwards (the captured one, ``-s 1 -c 1``)."""
    import torch
    import persistent_transformer_megakernel_gb300 as mk
    wl, s, _ = workload_desc(args.workload)
    w = W.make_weights(s, seed=0)
    dec = mk.Decoder(s, w, max_seq=64)
    dec.decode(W.make_prompt(s["vocab_in"], 16, seed=1), 0)
    dec.decode(None, 8)
    torch.cuda.synchronize()
    print("ncu case done: %s, 16 prompt forwards then 8 greedy forwards" % args.workload)


def prefill_case(args):
    """The prefill launch list's case: the workload's prompt through
    ``mk_prefill`` twice (only the last token's logits), device time printed."""
    import torch
    import persistent_transformer_megakernel_gb300 as mk
    wl, s, _ = workload_desc(args.workload)
    w = W.make_weights(s, seed=0)
    n = args.prefill_tokens if args.prefill_tokens > 0 else wl["prompt"]
    dec = mk.Decoder(s, w, max_seq=n + 8)
    prompt = torch.as_tensor(W.make_prompt(s["vocab_in"], n, seed=1), device="cuda")
    for rep in range(2):
        dec.reset()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        dec.prefill(prompt, all_ids=False)
        e1.record()
        e1.synchronize()
        print("prefill case %d: %s, %d-token prompt, %.3f ms" % (rep, args.workload, n, e0.elapsed_time(e1)))


def trace_case(args):
    """Phase times of the decode kernel from its %globaltimer stamps: the
    workload's prompt through ``mk_prefill``, then 64 traced greedy forwards."""
    import torch
    import persistent_transformer_megakernel_gb300 as mk
    from persistent_transformer_megakernel_gb300 import trace as T
    wl, s, desc = workload_desc(args.workload)
    if wl.get("sentinel"):
        raise SystemExit("--trace-case needs a workload with an id prompt")
    w = W.make_weights(s, seed=0)
    n = 64
    dec = mk.Decoder(s, w, max_seq=wl["prompt"] + n + 8)
    dec.prefill(W.make_prompt(s["vocab_in"], wl["prompt"], seed=1), all_ids=False)
    buf = T.buffer(dec, n)
    dec.decode(None, n, trace=buf)
    torch.cuda.synchronize()
    print("trace case: %s; %d greedy forwards after the prompt" % (desc, n))
    print(T.format_summary(T.summarize(buf, s["n_layers"])))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="mk", choices=["mk", "reference"])
    ap.add_argument("--workload", default="qwen3_0p6b", choices=sorted(W.WORKLOADS))
    ap.add_argument("--cpu-forwards", type=int, default=8)
    ap.add_argument("--ablation-forwards", type=int, default=32)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-ablation", action="store_true")
    ap.add_argument("--prefill-tokens", type=int, default=0,
                    help="prompt length of --prefill-case (default: the workload's prompt)")
    ap.add_argument("--prefill-case", action="store_true",
                    help="run the workload's prompt through mk_prefill twice (the prefill ncu launch list)")
    ap.add_argument("--trace-case", action="store_true",
                    help="print the decode kernel's per-phase times from its in-kernel stamps")
    ap.add_argument("--ncu-case", action="store_true",
                    help="run only the small profiling case (no JSON line)")
    args = ap.parse_args()
    if args.prefill_case:
        prefill_case(args)
        return
    if args.ncu_case:
        ncu_case(args)
        return
    if args.trace_case:
        trace_case(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and args.impl == "mk":
        import torch
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world)
    if world > 1 and args.impl == "mk":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
