#!/usr/bin/env python3
"""Paged decode-attention benchmark (one JSON line on rank 0).

A step is one pass of the decode hot path over one batch: the fork's
copy-on-write block copies (workloads that fork), then per layer the new
tokens' slot writes and the paged attention (split-K partitions + merge).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl pkv|reference]

``value`` is achieved HBM throughput of the step: algorithmic bytes (K/V of
the valid positions, q, out, block tables, lengths; slot writes; block
copies) per second, summed over ranks.  Pools are resident in HBM; the
replicas rotate so consecutive steps never reuse L2 contents.  ``e2e``
repeats the measurement through the public API with the step's inputs copied
from pinned host memory and the outputs read back every step.
``--impl reference`` times the CPU oracle on a bounded sample instead.
"""
import os

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import dataclasses
import hashlib
import json
import math
import re
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
import workloads as W  # noqa: E402

L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0
MIN_DECODE_EVENTS = 50         # CUDA-event samples behind the decode launch's median
METRIC = "paged decode attention: achieved HBM GB/s (% of GB300 peak); decode tokens/s"


# the measured configurations, by number, and the workload each one runs
CONFIGS = {1: "tiny", 2: "llama3_8b", 3: "llama2_70b_mixed_bs16", 4: "cow_fork", 5: "llama2_70b_step"}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    p.add_argument("--op", default="decode", choices=["decode", "swap", "verify"],
                   help="decode: the decode step (default); swap: preemption swap-out/in of a quarter of the "
                        "batch; verify: the multi-query (speculative verify) call")
    p.add_argument("--num-queries", type=int, default=4, help="query tokens per sequence for --op verify")
    p.add_argument("--workload", default="llama3_8b", choices=sorted(W.SPECS))
    p.add_argument("--config", type=int, choices=sorted(CONFIGS), default=None,
                   help="the measured configurations by number (1 tiny, 2 8B-shaped, 3 70B-shaped mixed, "
                        "4 copy-on-write forks, 5 80-layer 70B step); overrides --workload")
    p.add_argument("--block-size", type=int, choices=[16, 32], default=None,
                   help="with --config 3: the pool's block size (16 or 32)")
    p.add_argument("--dtype", choices=["f16", "bf16"], default=None,
                   help="16-bit type of q, out and the pools (default: the workload's own)")
    p.add_argument("--partition-tokens", type=int, default=0)
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="budget of the cpu_baseline sample")
    p.add_argument("--ref-seconds", type=float, default=90.0, help="total budget of the --impl reference run")
    p.add_argument("--layers", type=int, default=0,
                   help="run a multi-layer workload with this many layers (same per-layer shape; 0 = all)")
    p.add_argument("--separate-append", action="store_true",
                   help="launch paged_kv_append and the decode separately instead of the fused call")
    p.add_argument("--replicas", type=int, default=0,
                   help="pool replicas rotated between steps (0: enough to exceed L2; 1 for small profiler captures)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=200)
    p.add_argument("--e2e-eager", action="store_true",
                   help="end-to-end loop issues every call from Python instead of replaying a CUDA graph of the step")
    args = p.parse_args()
    if args.config is not None:
        args.workload = CONFIGS[args.config]
        if args.config == 3 and args.block_size == 32:
            args.workload = "llama2_70b_mixed_bs32"
    return args


def workload_spec(args) -> W.Spec:
    """The named workload, in the 16-bit type --dtype names when given."""
    spec = W.SPECS[args.workload]
    if args.dtype and args.dtype != spec.dtype:
        spec = dataclasses.replace(spec, dtype=args.dtype,
                                   description=f"{spec.description} (run in {args.dtype})")
    return spec


# ---------------------------------------------------------------- bytes
def algorithmic_bytes(wl: W.Workload) -> dict:
    """Algorithmic bytes of one step (one replica)."""
    s = wl.spec
    e, Hkv, Hq, d, bs = s.elem_bytes, s.num_kv_heads, s.num_heads, s.head_dim, s.block_size
    ekv = s.kv_elem_bytes                                  # 1 for an E4M3 pool
    L = wl.seq_lens.astype(np.int64)
    nb = (L + bs - 1) // bs
    small = 2 * s.num_seqs * Hq * d * e + 4 * int(nb.sum()) + 4 * s.num_seqs
    logical = int(2 * L.sum() * Hkv * d * ekv) + small
    # unique: each physical (block, slot) read once even if several sequences share it
    seen = {}
    for i in range(s.num_seqs):
        for j in range(int(nb[i])):
            b = int(wl.block_tables[i, j])
            seen[b] = max(seen.get(b, 0), min(bs, int(L[i]) - j * bs))
    unique = int(2 * sum(seen.values()) * Hkv * d * ekv) + small
    valid_tok = int((wl.slot_mapping >= 0).sum())
    append = 2 * valid_tok * Hkv * d * (e + ekv) + 8 * wl.num_tokens + (8 * Hkv if s.fp8 else 0)
    copy = 2 * 2 * len(wl.copy_pairs) * bs * Hkv * d * ekv * s.num_layers
    step = copy + s.num_layers * (append + unique)
    return dict(decode_unique=unique, decode_logical=logical, append=append, copy=copy, step=step)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def decode_source_hash() -> str:
    h = hashlib.sha256()
    for name in ("pkv_decode.cu", "pkv_decode_common.cuh", "pkv_decode_plan.cu", "pkv_device.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_156_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def verify_source_hash() -> str:
    h = hashlib.sha256()
    for name in ("pkv_verify_tc.cu", "pkv_tcgen05.cuh", "pkv_decode_common.cuh", "pkv_decode_plan.cu", "pkv_device.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_156_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_verify_traffic(workload: str, num_queries: int, fp8: bool = False):
    """Per-launch DRAM bytes of the verify kernel from the committed ncu summary for
    this workload and query count, or None (no summary, or the sources changed).  An
    E4M3 pool's verify runs the decode kernel's multi-query form: its sources decide."""
    path = os.path.join(ROOT, "profiles", f"verify_{workload}_nq{num_queries}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_t = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    m_h = re.search(r"(?:verify|decode)_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m_t or not m_h or m_h.group(1) != (decode_source_hash() if fp8 else verify_source_hash()):
        return None
    return int(m_t.group(1))


def profiled_traffic(workload: str):
    """Per-launch DRAM bytes of the decode kernel from the committed ncu summary,
    or None when there is none or the kernel source changed since the capture."""
    path = os.path.join(ROOT, "profiles", f"decode_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_t = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    m_h = re.search(r"decode_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m_t or not m_h or m_h.group(1) != decode_source_hash():
        return None
    return int(m_t.group(1))


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu_index = gpu_index
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(gpu_index), "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for i, n in enumerate(names):
                if r[5 + i].strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------- oracle timing
def time_oracle(wl: W.Workload, pools, seqs, budget_s: float):
    """Run the oracle (slot writes, then attention) for sequences in ``seqs``,
    cycling until ``budget_s`` has elapsed; returns (bytes, seconds, sequences)."""
    import oracle

    spec = wl.spec
    kc, vc = pools
    tok_of = {}
    # the appended tokens of each sequence, in slot_mapping order
    t = 0
    for s in range(spec.num_seqs):
        n = 1
        if spec.fork is not None:
            L, P = int(wl.seq_lens[s]), spec.fork[2]
            Pc = W.blocks_needed(P, spec.block_size) * spec.block_size
            n = max(1, len(set(range(P, min(L, Pc))) | ({L - 1} if L > P else set())))
        tok_of[s] = list(range(t, t + n))
        t += n
    per = algorithmic_bytes(wl)
    Hkv, d, e, ekv = spec.num_kv_heads, spec.head_dim, spec.elem_bytes, spec.kv_elem_bytes
    done_bytes, done = 0, 0
    t0 = time.perf_counter()
    i = 0
    while True:
        s = seqs[i % len(seqs)]
        idx = tok_of[s]
        if spec.fp8:
            ks, vs = wl.k_scales[0], wl.v_scales[0]
            oracle.append_fp8_ref(kc, vc, wl.k_new[idx], wl.v_new[idx], wl.slot_mapping[idx], ks, vs, spec.dtype)
            oracle.attention_fp8_ref(wl.q[s:s + 1], kc, vc, wl.block_tables[s:s + 1], wl.seq_lens[s:s + 1], wl.scale,
                                     Hkv, spec.dtype, ks, vs)
        else:
            oracle.append_ref(kc, vc, wl.k_new[idx], wl.v_new[idx], wl.slot_mapping[idx])
            oracle.attention_ref(wl.q[s:s + 1], kc, vc, wl.block_tables[s:s + 1], wl.seq_lens[s:s + 1], wl.scale, Hkv,
                                 spec.dtype)
        L = int(wl.seq_lens[s])
        done_bytes += 2 * L * Hkv * d * ekv + 2 * spec.num_heads * d * e + 4 * W.blocks_needed(L, spec.block_size) + 4
        done_bytes += 2 * len(idx) * Hkv * d * (e + ekv) + 8 * len(idx)
        done += 1
        i += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    del per
    return done_bytes, time.perf_counter() - t0, done


def sample_for_oracle(wl: W.Workload, n: int = 16):
    rng = np.random.default_rng(99)
    return sorted(rng.choice(wl.spec.num_seqs, size=min(n, wl.spec.num_seqs), replace=False).tolist())


# ---------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- the library arm
def run_pkv(args, rank, world, local):
    from paged_kv_cache_156_gb300 import _build

    if local == 0:
        _build.build()
    barrier(world)
    import paged_kv_cache_156_gb300 as pkv

    pkv.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    spec = workload_spec(args)
    if args.layers and spec.num_layers > 1:
        spec = dataclasses.replace(spec, num_layers=min(args.layers, spec.num_layers))
    wl = W.build(spec, values="none")
    tdt = torch.float16 if spec.dtype == W.F16 else torch.bfloat16
    nbytes = algorithmic_bytes(wl)

    def dev_bits(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(tdt)

    q, k_new, v_new = dev_bits(wl.q), dev_bits(wl.k_new), dev_bits(wl.v_new)
    slots = torch.from_numpy(wl.slot_mapping).to(dev)
    tables = torch.from_numpy(wl.block_tables).to(dev)
    lens = torch.from_numpy(wl.seq_lens).to(dev)
    pairs = torch.from_numpy(wl.copy_pairs).to(dev)
    footprint = wl.pool_bytes_per_layer() * spec.num_layers
    replicas = max(2, min(4, math.ceil(3 * L2_BYTES / footprint))) if spec.num_layers == 1 else 1
    if footprint * replicas > 0.6 * torch.cuda.get_device_properties(dev).total_memory:
        replicas = 1
    if args.replicas > 0:
        replicas = args.replicas
    pools = []
    for r in range(replicas):
        kcs, vcs = [], []
        for l in range(spec.num_layers):
            k, v = W.device_pools(wl, l, dev)
            kcs.append(k)
            vcs.append(v)
        pools.append((kcs, vcs))
    outs = [torch.empty_like(q) for _ in range(spec.num_layers)]
    k_scales = [torch.from_numpy(x).to(dev) for x in wl.k_scales]      # E4M3 pools only
    v_scales = [torch.from_numpy(x).to(dev) for x in wl.v_scales]
    # 0 = automatic: the host sizes the workspace for the smallest partition,
    # the plan kernel picks the size from the lengths
    part_min = args.partition_tokens or pkv.decode_partition_tokens(spec.num_seqs, spec.num_heads,
                                                                    spec.num_kv_heads, spec.head_dim, wl.max_seq_len)
    ws = pkv.alloc_workspace(spec.num_seqs, spec.num_heads, spec.num_kv_heads, spec.head_dim, wl.max_seq_len,
                             args.partition_tokens, dev)
    planned = spec.num_seqs <= pkv.PLAN_MAX_SEQS
    max_parts_min = math.ceil(wl.max_seq_len / part_min) if wl.max_seq_len else 1
    # A step plans once (the batch is the same in every layer: lengths and block tables do not
    # depend on this step's slot writes); every layer then writes its new tokens and decodes over
    # the plan.  With one new token per sequence (decode proper) the slot write rides in the decode
    # launch (pkv_paged_kv_append_decode); a step that writes more slots per sequence (the rest of a
    # copied block) launches paged_kv_append first.  The decode events time the decode kernel
    # alone; the step value counts the plan too.
    fused = wl.num_tokens == spec.num_seqs and not args.separate_append
    launches_per_step = (1 if len(wl.copy_pairs) else 0) + (1 if planned else 0) + spec.num_layers * (
        (1 if fused else 2) + (0 if planned or max_parts_min == 1 else 1))

    total_len = int(wl.seq_lens.sum())             # the scheduler knows it; it sizes the decode grid
    ev_pairs = []
    copy_ev = []                                    # copy-on-write copies, timed apart from the decode

    def step(i, timed):
        kcs, vcs = pools[i % replicas]
        if len(wl.copy_pairs):
            if timed:
                ca = torch.cuda.Event(enable_timing=True)
                ca.record()
            pkv.copy_blocks(kcs, vcs, pairs)
            if timed:
                cb = torch.cuda.Event(enable_timing=True)
                cb.record()
                copy_ev.append((ca, cb))
        if fused:
            pkv.decode_plan(ws, tables, lens, spec.num_heads, kcs[0], wl.max_seq_len, args.partition_tokens,
                            sum_seq_lens=total_len)
        for l in range(spec.num_layers):
            if not fused:
                if spec.fp8:
                    pkv.paged_kv_append_fp8(k_new, v_new, kcs[l], vcs[l], slots, k_scales[l], v_scales[l])
                else:
                    pkv.paged_kv_append(k_new, v_new, kcs[l], vcs[l], slots)
                if l == 0:
                    pkv.decode_plan(ws, tables, lens, spec.num_heads, kcs[0], wl.max_seq_len, args.partition_tokens,
                                    sum_seq_lens=total_len)
            # decode events: around layer 0's launch, or, for a fused multi-layer step, around
            # layers 1 .. L-1 (back-to-back decode launches, nothing else in between)
            chain = fused and spec.num_layers > 1
            rec = timed and (l == 0 if not chain else l == spec.num_layers - 1)
            if timed and (l == 0 if not chain else l == 1):
                a = torch.cuda.Event(enable_timing=True)
                a.record()
            kw = dict(scale=wl.scale, max_seq_len=wl.max_seq_len, workspace=ws, partition_tokens=args.partition_tokens,
                      planned=True, sum_seq_lens=total_len)
            if fused:
                if spec.fp8:
                    kw.update(k_scale=k_scales[l], v_scale=v_scales[l])
                # layers after the first: nothing pending writes their pools, the tables or the
                # plan (the preceding launch is the previous layer's), so their tile loads may
                # start while it finishes
                pkv.paged_kv_append_decode(outs[l], q, k_new, v_new, kcs[l], vcs[l], slots, tables, lens,
                                           inputs_ready=l > 0, **kw)
            elif spec.fp8:
                pkv.paged_attention_decode_fp8(outs[l], q, kcs[l], vcs[l], tables, lens, k_scales[l], v_scales[l], **kw)
            else:
                pkv.paged_attention_decode(outs[l], q, kcs[l], vcs[l], tables, lens, **kw)
            if rec:
                b = torch.cuda.Event(enable_timing=True)
                b.record()
                ev_pairs.append((a, b))

    for i in range(max(3, args.warmup)):
        step(i, False)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0, "device error word raised during warm-up"
    part = pkv.decode_plan_partition_tokens(ws, spec.num_seqs, spec.num_heads, spec.num_kv_heads) if planned \
        else part_min
    max_parts = math.ceil(wl.max_seq_len / part) if wl.max_seq_len else 1

    clocks = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(args.steps):
        step(i, True)
    t1.record()
    torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = t0.elapsed_time(t1)
    # the decode launch's median needs at least MIN_DECODE_EVENTS samples: steps
    # past the timed region (not in `value`) add events when K is smaller
    n_timed_events = len(ev_pairs)
    for i in range(max(0, MIN_DECODE_EVENTS - n_timed_events)):
        step(args.steps + i, True)
    torch.cuda.synchronize()
    clk = clocks.stop()
    max_ms = max_over_ranks(elapsed_ms, world)
    dec_launches = spec.num_layers - 1 if (fused and spec.num_layers > 1) else 1
    dec_ms = float(np.median([a.elapsed_time(b) for a, b in ev_pairs])) / dec_launches
    assert pkv.device_error() == 0, "device error word raised during the timed region"

    value = world * nbytes["step"] * args.steps / (max_ms / 1e3) / 1e9
    peak, peak_kind = load_peaks()
    # the timed launch moves the decode's bytes, plus the slot write's when it is fused in
    kernel_bytes = nbytes["decode_unique"] + (nbytes["append"] if fused else 0)
    dec_gbs = kernel_bytes / (dec_ms / 1e3) / 1e9
    traffic = profiled_traffic(args.workload)
    copy = None
    if copy_ev:                                     # the step's copy_blocks launch on its own
        copy_ms = float(np.median([a.elapsed_time(b) for a, b in copy_ev]))
        copy = {"kernel": "copy_blocks_kernel", "pairs": int(len(wl.copy_pairs)), "layers": spec.num_layers,
                "algorithmic_bytes_per_launch": nbytes["copy"], "avg_launch_ms": round(copy_ms, 5),
                "achieved": round(nbytes["copy"] / (copy_ms / 1e3) / 1e9, 2), "unit": "GB/s",
                "frac": round(nbytes["copy"] / (copy_ms / 1e3) / 1e9 / peak, 4), "launch_events": len(copy_ev)}

    # ---- end to end: inputs from pinned host memory, outputs read back, every step
    def measure_e2e(use_graph):
        host_in = [t.cpu().pin_memory() for t in (q, k_new, v_new, slots, tables, lens)]
        dev_in = [q, k_new, v_new, slots, tables, lens]
        # two pinned output buffers: the host reads step i-1's outputs while the GPU runs step i
        host_out = [[torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs] for _ in range(2)]
        done = [torch.cuda.Event(), torch.cuda.Event()]
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out[0])
        n_e2e = max(3, args.e2e_steps)
        seen = 0.0

        def read_result(buf):                        # the host uses the step's result
            return float(buf[0].view(-1)[0].float()) + float(buf[-1].view(-1)[-1].float())

        def whole_step(i, j):                    # inputs in, the step, outputs out
            for h, d_ in zip(host_in, dev_in):
                d_.copy_(h, non_blocking=True)
            step(i, False)
            for h, o in zip(host_out[j], outs):
                h.copy_(o, non_blocking=True)

        graphs = None
        if use_graph:
            # one CUDA graph per (pool replica, output buffer), captured through the same
            # public calls; a replay copies the inputs in, plans, decodes and copies the
            # outputs back, with one launch from the host
            torch.cuda.synchronize()
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                for r in range(replicas):
                    whole_step(r, 0)
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            graphs = {}
            for r in range(replicas):
                for j in range(2):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, capture_error_mode="relaxed"):
                        whole_step(r, j)
                    graphs[(r, j)] = g
            torch.cuda.synchronize()
            assert pkv.device_error() == 0, "device error word raised while capturing"
        else:
            for i in range(3):                   # warm the eager path's host side
                whole_step(i, i % 2)

        torch.cuda.synchronize()
        barrier(world)
        w0 = time.perf_counter()
        for i in range(n_e2e):
            j = i % 2
            if graphs is not None:
                graphs[(i % replicas, j)].replay()
            else:
                whole_step(i, j)
            done[j].record()
            if i > 0:
                done[1 - j].synchronize()
                seen += read_result(host_out[1 - j])
        done[(n_e2e - 1) % 2].synchronize()
        seen += read_result(host_out[(n_e2e - 1) % 2])
        e2e_s = max_over_ranks(time.perf_counter() - w0, world)
        return {"value": round(world * nbytes["step"] * n_e2e / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": n_e2e,
                "ms_per_step": round(e2e_s * 1e3 / n_e2e, 4),
                "pipeline": ("every step copies its inputs in from pinned memory and its outputs back; the host "
                             "reads step i's outputs while the GPU runs step i+1; " +
                             ("each step is one replay of a CUDA graph of the public calls"
                              if graphs is not None else
                              "every call issued from Python through the C ABI (host validation and "
                              "launch set-up on every step)")),
                "finite": bool(math.isfinite(seen))}

    e2e = e2e_eager = None
    if not args.no_e2e:
        e2e = measure_e2e(not args.e2e_eager)
        if not args.e2e_eager:
            e2e_eager = measure_e2e(False)

    # ---- CPU oracle on a bounded sample (rank 0, one GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if spec.fp8:
            kc0 = pools[0][0][0].cpu().numpy().copy()
            vc0 = pools[0][1][0].cpu().numpy().copy()
        else:
            kc0 = pools[0][0][0].contiguous().view(torch.int16).cpu().numpy().view(np.uint16).copy()
            vc0 = pools[0][1][0].contiguous().view(torch.int16).cpu().numpy().view(np.uint16).copy()
        seqs = sample_for_oracle(wl)
        b, sec, n = time_oracle(wl, (kc0, vc0), seqs, args.cpu_seconds)
        cpu = {"value": round(b / sec / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} sequence decodes (slot writes + attention, layer 0) cycling over {len(seqs)} "
                         f"sequences of the workload, {sec:.1f} s single-threaded float64 numpy",
               "nproc": os.cpu_count()}

    if rank != 0:
        return None
    return {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(max_ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": spec.dtype,
        "data": "synthetic (seeded N(0,1) K/V/q, permuted block pools)",
        "config": {"workload": spec.name, "description": spec.description, "num_seqs": spec.num_seqs,
                   "num_heads": spec.num_heads, "num_kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim,
                   "block_size": spec.block_size, "num_layers": spec.num_layers,
                   "kv_dtype": spec.kv_dtype or spec.dtype,
                   "mean_seq_len": round(float(wl.seq_lens.mean()), 1), "max_seq_len": wl.max_seq_len,
                   "num_blocks": wl.num_blocks, "copy_pairs": int(len(wl.copy_pairs)),
                   "partition_tokens": part, "partition_tokens_min": part_min, "max_partitions": max_parts,
                   "work_list": "plan kernel" if planned else "full grid",
                   "slot_write": "fused into the decode launch" if fused else "paged_kv_append launch",
                   "l2": f"inputs larger than L2: {replicas} rotating pool replicas of "
                         f"{footprint / 1e9:.3f} GB each (L2 {L2_BYTES / 2**20:.0f} MiB)",
                   "parallelism": f"replicas x{world} (no data-path collective)"},
        "tokens_per_s": round(world * spec.num_seqs * args.steps / (max_ms / 1e3), 1),
        "step_bytes": nbytes,
        "roofline": {"bound": "hbm", "kernel": ("decode_kernel (" +
                                                (f"mean of layers 1..{spec.num_layers - 1}, launched back to back"
                                                 if dec_launches > 1 else "planned run of layer 0") +
                                                ", in-kernel split-K merge" +
                                                (", slot write fused in" if fused else "") +
                                                "; the step's one plan kernel is outside this timing, inside value)"),
                     "achieved": round(dec_gbs, 2), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(dec_gbs / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": kernel_bytes, "avg_launch_ms": round(dec_ms, 5),
                     "launch_events": len(ev_pairs), "launch_events_in_timed_region": n_timed_events},
        "copy_blocks": copy,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "e2e_eager": e2e_eager,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }


# ---------------------------------------------------------------- the reference arm (CPU oracle)
def run_reference(args, rank, world):
    if rank != 0:
        return None
    spec = workload_spec(args)
    wl = W.build(spec, values="none")
    seqs = sample_for_oracle(wl, 4)
    pools = W.host_pools_for(wl, seqs, 0)
    # size each step: time one sequence, then give each step ~budget/(K+W)
    b1, s1, _ = time_oracle(wl, [np.array(x, copy=True) for x in pools], seqs[:1], 0.0)
    per_step_s = min(5.0, max(s1, args.ref_seconds / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        time_oracle(wl, pools, seqs, per_step_s)
    tot_b, tot_s, tot_n = 0, 0.0, 0
    for _ in range(args.steps):
        b, s, n = time_oracle(wl, pools, seqs, per_step_s)
        tot_b += b
        tot_s += s
        tot_n += n
    value = tot_b / tot_s / 1e9
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tot_s * 1e3 / max(1, args.steps), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype,
            "data": "synthetic (seeded N(0,1), sampled sequences)",
            "config": {"workload": spec.name, "description": spec.description},
            "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "kind": "oracle", "cores": 1,
                             "sample": f"{tot_n} sequence decodes over {len(seqs)} sampled sequences, "
                                       f"~{per_step_s:.2f} s per step, float64 numpy single-threaded",
                             "nproc": os.cpu_count()},
            "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------- swap (preemption) measurement
def run_swap(args, rank, world, local):
    """Swap a quarter of the batch's sequences out to pinned host pools and back in.

    One step = swap-out (device -> pinned host) then swap-in (host -> device,
    new block ids) of every block those sequences use, all layers.  Bytes are
    the K and V bytes of the swapped blocks, counted once per direction.
    """
    from paged_kv_cache_156_gb300 import _build

    if local == 0:
        _build.build()
    barrier(world)
    import paged_kv_cache_156_gb300 as pkv

    pkv.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    spec = workload_spec(args)
    wl = W.build(spec, values="none")
    tdt = torch.float16 if spec.dtype == W.F16 else torch.bfloat16
    bs = spec.block_size
    seqs = list(range(0, spec.num_seqs, 4))
    used = np.unique(np.concatenate([wl.block_tables[s, :W.blocks_needed(int(wl.seq_lens[s]), bs)] for s in seqs]))
    nb = len(used)
    layers = spec.num_layers
    kcs, vcs = [], []
    for l in range(layers):
        k, v = W.device_pools(wl, l, dev)
        kcs.append(k)
        vcs.append(v)
    shape = (nb,) + tuple(kcs[0].shape[1:])
    hk = [torch.empty(shape, dtype=tdt, pin_memory=True) for _ in range(layers)]
    hv = [torch.empty(shape, dtype=tdt, pin_memory=True) for _ in range(layers)]
    free = np.setdiff1d(np.arange(wl.num_blocks), used)
    back = np.concatenate([free, used])[:nb]
    out_pairs = torch.from_numpy(np.stack([used, np.arange(nb)], 1).astype(np.int64)).to(dev)
    in_pairs = torch.from_numpy(np.stack([np.arange(nb), back], 1).astype(np.int64)).to(dev)
    block_bytes = 2 * bs * spec.num_kv_heads * spec.head_dim * 2 * layers     # K and V, all layers
    ev = []

    def step(timed):
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record()
        pkv.swap_blocks(kcs, vcs, hk, hv, out_pairs)
        b.record()
        pkv.swap_blocks(hk, hv, kcs, vcs, in_pairs)
        c.record()
        if timed:
            ev.append((a, b, c))

    for _ in range(max(3, args.warmup)):
        step(False)
    torch.cuda.synchronize()
    barrier(world)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        step(True)
    t1.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1), world)
    assert pkv.device_error() == 0
    out_ms = float(np.mean([a.elapsed_time(b) for a, b, _ in ev]))
    in_ms = float(np.mean([b.elapsed_time(c) for _, b, c in ev]))
    step_bytes = 2 * nb * block_bytes
    # the link's roofline: the copy engines moving the same bytes between one
    # contiguous pinned buffer and one device buffer (cudaMemcpyAsync via torch)
    hbuf = torch.empty(nb * block_bytes, dtype=torch.uint8, pin_memory=True)
    dbuf = torch.empty(nb * block_bytes, dtype=torch.uint8, device=dev)
    ce = []
    for i in range(max(3, args.warmup) + args.steps):
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record()
        hbuf.copy_(dbuf, non_blocking=True)
        b.record()
        dbuf.copy_(hbuf, non_blocking=True)
        c.record()
        if i >= max(3, args.warmup):
            ce.append((a, b, c))
    torch.cuda.synchronize()
    ce_out = float(np.mean([a.elapsed_time(b) for a, b, _ in ce]))
    ce_in = float(np.mean([b.elapsed_time(c) for _, b, c in ce]))
    ce_gbs = 2 * nb * block_bytes / ((ce_out + ce_in) / 1e3) / 1e9
    if rank != 0:
        return None
    return {"metric": "swap_blocks: device <-> pinned host GB/s (swap-out then swap-in)",
            "value": round(world * step_bytes * args.steps / (ms / 1e3) / 1e9, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": spec.dtype,
            "data": "synthetic", "config": {"workload": spec.name, "swapped_sequences": len(seqs), "blocks": int(nb),
                                            "bytes_per_direction": int(nb * block_bytes), "layers": layers},
            "swap_out_GBps": round(nb * block_bytes / (out_ms / 1e3) / 1e9, 2),
            "swap_in_GBps": round(nb * block_bytes / (in_ms / 1e3) / 1e9, 2),
            "roofline": {"bound": "link", "achieved": round(step_bytes / ((out_ms + in_ms) / 1e3) / 1e9, 2),
                         "peak": round(ce_gbs, 2), "peak_kind": "measured: copy engines, same bytes, contiguous",
                         "unit": "GB/s", "frac": round(step_bytes / ((out_ms + in_ms) / 1e3) / 1e9 / ce_gbs, 4),
                         "copy_engine_out_GBps": round(nb * block_bytes / (ce_out / 1e3) / 1e9, 2),
                         "copy_engine_in_GBps": round(nb * block_bytes / (ce_in / 1e3) / 1e9, 2),
                         "traffic": None},   # bounded by the host link, not by DRAM: no ncu DRAM figure applies
            "gpu_launches": 2 * args.steps * ((layers + 63) // 64)}


def run_verify(args, rank, world, local):
    """The multi-query verify call: num_queries query tokens per sequence, causal
    among themselves, over the workload's paged K/V (the last num_queries
    positions of each sequence are the query tokens' own).  Bytes: K/V of every
    valid position once, plus q and out."""
    from paged_kv_cache_156_gb300 import _build

    if local == 0:
        _build.build()
    barrier(world)
    import paged_kv_cache_156_gb300 as pkv

    pkv.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    spec = workload_spec(args)
    if spec.num_layers != 1:
        raise SystemExit("--op verify runs single-layer workloads")
    wl = W.build(spec, values="none")
    tdt = torch.float16 if spec.dtype == W.F16 else torch.bfloat16
    nq = args.num_queries
    B, Hq, d = spec.num_seqs, spec.num_heads, spec.head_dim
    g = torch.Generator(device=dev)
    g.manual_seed(spec.seed)
    q = torch.randn((B, nq, Hq, d), generator=g, device=dev, dtype=torch.float32).to(tdt)
    out = torch.empty_like(q)
    tables = torch.from_numpy(wl.block_tables).to(dev)
    lens_h = np.maximum(wl.seq_lens, nq)
    lens = torch.from_numpy(lens_h).to(dev)
    total_len = int(lens_h.sum())                   # sizes the grid
    footprint = wl.pool_bytes_per_layer()
    replicas = max(2, min(4, math.ceil(3 * L2_BYTES / footprint)))
    pools = [W.device_pools(wl, 0, dev) for _ in range(replicas)]
    k_new = torch.from_numpy(np.ascontiguousarray(wl.k_new).view(np.int16)).to(dev).view(tdt)
    v_new = torch.from_numpy(np.ascontiguousarray(wl.v_new).view(np.int16)).to(dev).view(tdt)
    slots = torch.from_numpy(wl.slot_mapping).to(dev)
    scales = {}
    if spec.fp8:                                    # E4M3 pools: per-KV-head scales
        scales = dict(k_scale=torch.from_numpy(wl.k_scales[0]).to(dev), v_scale=torch.from_numpy(wl.v_scales[0]).to(dev))
    for k, v in pools:                               # the step's new tokens, so every position holds one
        if spec.fp8:
            pkv.paged_kv_append_fp8(k_new, v_new, k, v, slots, scales["k_scale"], scales["v_scale"])
        else:
            pkv.paged_kv_append(k_new, v_new, k, v, slots)
    ws = pkv.alloc_workspace(B, Hq * nq, spec.num_kv_heads, d, wl.max_seq_len, args.partition_tokens, dev)
    nbytes = algorithmic_bytes(wl)["decode_unique"] + 2 * B * (nq - 1) * Hq * d * spec.elem_bytes

    def call(i):
        k, v = pools[i % replicas]
        pkv.paged_attention_verify(out, q, k, v, tables, lens, wl.scale, max_seq_len=wl.max_seq_len, workspace=ws,
                                   partition_tokens=args.partition_tokens, sum_seq_lens=total_len, **scales)

    for i in range(max(3, args.warmup)):
        call(i)
    torch.cuda.synchronize()
    assert pkv.device_error() == 0
    barrier(world)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(args.steps):
        call(i)
    t1.record()
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1), world)
    assert pkv.device_error() == 0
    part = pkv.decode_plan_partition_tokens(ws, B, Hq * nq, spec.num_kv_heads) if B <= pkv.PLAN_MAX_SEQS else -1
    if rank != 0:
        return None
    gbs = world * nbytes * args.steps / (ms / 1e3) / 1e9
    peak, peak_kind = load_peaks()
    return {"metric": "paged verify attention GB/s (K/V of valid positions + q/out)", "value": round(gbs, 2),
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms / args.steps, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": spec.dtype, "data": "synthetic",
            "config": {"workload": spec.name, "num_queries": nq, "partition_tokens": part,
                       "l2": f"{replicas} rotating pool replicas"},
            "roofline": {"bound": "hbm", "achieved": round(gbs / world, 2), "peak": peak, "peak_kind": peak_kind,
                         "unit": "GB/s", "frac": round(gbs / world / peak, 4),
                         "traffic": profiled_verify_traffic(spec.name, nq, spec.fp8),
                         "algorithmic_bytes_per_launch": int(nbytes)},
            "gpu_launches": 2 * args.steps}


def main():
    args = parse_args()
    rank, world, local = dist_setup(args)
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    elif args.op == "swap":
        res = run_swap(args, rank, world, local)
    elif args.op == "verify":
        res = run_verify(args, rank, world, local)
    else:
        res = run_pkv(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
