"""Benchmark: decode attention over a packed INT4/INT2 KV cache on GB300.

One step = one kvq_decode_attn call (every hot-path stage: packed-tile loads,
operand construction, QK^T and PV tensor-core MMAs, affine folds, online
softmax, split merge) over the whole batch, with the packed cache resident in
HBM.  The metric is the effective KV-access bandwidth: packed K and V codes
plus their fp16 scales and offsets, divided by the step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kvq|reference]
                  [--workload NAME] [--no-extra]

--impl reference times the CPU oracle (the plain fp64 definition, not tuned)
on a bounded sample of the same workload.  Under torchrun (N > 1) every rank
runs its own replica of the per-GPU workload (weak scaling, no collective in
the data path); timings are max-reduced over ranks and rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
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

import torch  # noqa: E402

import kvq_synth as synth  # noqa: E402

DEFAULT_WORKLOAD = "b128_l32k_int4"
FALLBACK_HBM_GBS = 6800.0
SCHEME_NAMES = {0: "token", 1: "channel"}


# ----------------------------------------------------------------- set-up
def algorithmic_bytes(w, lens) -> int:
    """Packed K+V codes and their fp16 scale/offset arrays touched by a step."""
    blocks = sum((int(n) + 127) // 128 for n in lens) * w.num_kv_heads
    return blocks * block_bytes_kv(w)


def block_bytes_kv(w) -> int:
    """K and V codes of one 128-token block of one KV head, plus their fp16
    s and z (128 * D / G values each)."""
    return 2 * (128 * w.head_dim * w.bits // 8) + 2 * 2 * (128 * w.head_dim // w.group) * 2


def build_cache(w, seed, dev, k_scheme=None, v_scheme=None, chunk=16):
    """Pack K and V of a workload on the GPU, a few sequences at a time."""
    import bit_quantized_kv_decode_gb300 as kvq
    ks = w.k_scheme if k_scheme is None else k_scheme
    vs = w.v_scheme if v_scheme is None else v_scheme
    lens = synth.seq_lens_for(w, seed)
    max_blocks = (int(lens.max()) + 127) // 128
    if w.paged:
        pt_cpu, num_pages = synth.page_table_for(lens, seed, max_blocks)
        pt = pt_cpu.to(dev)
    else:
        pt, num_pages = None, w.batch * max_blocks
    desc = kvq.cache_desc(w.bits, ks, vs, w.num_kv_heads, num_pages, head_dim=w.head_dim, group=w.group)
    kc, vc = kvq.alloc_cache(desc, dev), kvq.alloc_cache(desc, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    cs = synth.outlier_channels(w, seed, dev)
    for b0 in range(0, w.batch, chunk):
        b1 = min(w.batch, b0 + chunk)
        sub_lens = lens[b0:b1]
        L = int(sub_lens.max())
        for which, cache in ((0, kc), (1, vc)):
            x = torch.zeros(b1 - b0, w.num_kv_heads, L, w.head_dim, device=dev)
            for b in range(b0, b1):
                for h in range(w.num_kv_heads):
                    n = int(lens[b])
                    x[b - b0, h, :n] = synth.kv_unit(w, seed, which, b, h, n, dev,
                                                     cs[h] if which == 0 else None)
            if pt is not None:
                sub_pt = pt[b0:b1].contiguous()
            else:
                sub_pt = (torch.arange(b0 * max_blocks, b1 * max_blocks, dtype=torch.int32, device=dev)
                          .view(b1 - b0, max_blocks))
            kvq.pack(desc, which, x, sub_lens.to(dev), sub_pt, cache=cache, dev_status=status)
            del x
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"pack reported device status {int(status.item()):#x}")
    q = synth.query(w, seed, dev)
    return dict(desc=desc, k=kc, v=vc, q=q, lens=lens.to(dev), lens_cpu=lens, pt=pt, max_blocks=max_blocks)


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        sel = [p for t, p in self.samples if t0 - 0.25 <= t <= t1 + 0.25] or [p for _, p in self.samples[-3:]]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in sel if num(p[1]) is not None]
        mx = [num(p[2]) for p in sel if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in sel for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sel)}


# ------------------------------------------------------------------ timing
def time_steps(fn, steps: int, warmup: int, stream):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    per = [a.elapsed_time(b) for a, b in ev]
    return sum(per) / len(per), per


L2_BYTES = 129 * 1024 * 1024


def rotation_sets(w, seed) -> int:
    """Cache copies a timed loop rotates through so that consecutive steps
    never find their inputs in the 129 MB L2 (1 when a step alone streams
    more than the L2 holds)."""
    per_step = algorithmic_bytes(w, synth.seq_lens_for(w, seed).tolist())
    return 1 if per_step > L2_BYTES else max(8, -(-2 * L2_BYTES // per_step))


KERNEL_SPECIALISED = "kvq::decode_kernel"
KERNEL_GENERAL = "kvq::decode_general_kernel (+ plan and merge kernels)"
SPLIT_SPECIALISED = "persistent CTAs cut the tile order into equal ranges; cut units are merged in the kernel"
SPLIT_GENERAL = ("a plan kernel cuts each unit's blocks into ranges in proportion to its sequence's length; "
                 "one range per CTA; a log-sum-exp merge kernel combines the ranges")


def measure_kvq(w, seed, steps, warmup, dev, k_scheme=None, v_scheme=None, e2e=True, mode=0, sets=None, flags=0):
    import bit_quantized_kv_decode_gb300 as kvq
    sets = rotation_sets(w, seed) if sets is None else sets
    # every copy holds the same inputs (the same seed): only the addresses differ
    cs = [build_cache(w, seed, dev, k_scheme, v_scheme) for _ in range(sets)]
    c = cs[0]
    desc = c["desc"]
    ad = kvq.attn_desc(desc, w.batch, c["max_blocks"], mode=mode, num_q_heads=w.num_q_heads, flags=flags)
    ws = torch.empty(kvq.workspace_size(ad), dtype=torch.uint8, device=dev)
    out = torch.empty(w.batch, w.num_q_heads, w.head_dim, dtype=torch.float32, device=dev)
    lse = torch.empty(w.batch, w.num_q_heads, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    turn = [0]

    def step():
        ci = cs[turn[0] % sets]
        turn[0] += 1
        kvq.decode_attn(desc, ci["q"], ci["k"], ci["v"], ci["lens"], ci["pt"], ci["max_blocks"], mode=mode, out=out,
                        lse=lse, workspace=ws, dev_status=status, flags=flags)

    t_wall0 = time.time()
    ms, per = time_steps(step, steps, warmup, stream)
    t_wall1 = time.time()
    if int(status.item()) != 0:
        raise RuntimeError(f"decode reported device status {int(status.item()):#x}")
    general = kvq.decode_path(ad) == kvq._lib.PATH_GENERAL  # plan, block-range and log-sum-exp merge kernels
    res = dict(ms=ms, per=per, bytes=algorithmic_bytes(w, c["lens_cpu"].tolist()), t0=t_wall0, t1=t_wall1,
               launches=steps * (3 if general else 1), sets=sets, lens=c["lens_cpu"].tolist(), general=general,
               kernel=KERNEL_GENERAL if general else KERNEL_SPECIALISED)
    if e2e:
        # end to end through the public API with host buffers: H2D of this step's
        # query and lengths from pinned memory, decode, D2H of out and lse
        q_h = c["q"].cpu().pin_memory()
        lens_h = c["lens_cpu"].clone().pin_memory()
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        q_d = torch.empty_like(c["q"])
        lens_d = torch.empty_like(c["lens"])

        def e2e_step():
            q_d.copy_(q_h, non_blocking=True)
            lens_d.copy_(lens_h, non_blocking=True)
            kvq.decode_attn(desc, q_d, c["k"], c["v"], lens_d, c["pt"], c["max_blocks"], mode=mode, out=out, lse=lse,
                            workspace=ws, dev_status=status)
            out_h.copy_(out, non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)

        e2e_ms, _ = time_steps(e2e_step, max(1, steps // 2), max(3, warmup), stream)
        res.update(e2e_ms=e2e_ms, h2d=q_h.numel() * 2 + lens_h.numel() * 4,
                   d2h=out_h.numel() * 4 + lse_h.numel() * 4)
    del c, cs
    torch.cuda.empty_cache()
    return res


def l2_note(res) -> str:
    if res["sets"] > 1:
        return ("each step reads %.1f MB (< 129 MB L2): timed steps rotate over %d cache copies "
                "(%.0f MB), so no step finds its inputs in L2" % (res["bytes"] / 1e6, res["sets"],
                                                                  res["sets"] * res["bytes"] / 1e6))
    return "each step reads %.2f GB > 129 MB L2; no flush needed" % (res["bytes"] / 1e9)


# ------------------------------------------------------------ CPU oracle
def _oracle_unit(args):
    """Oracle decode of one (sequence, kv head) from its packed blocks: unpack,
    dequantize, attend (the CPU definition, as it stands)."""
    import numpy as np
    from oracle import kvq_oracle as orc
    (q_bits, kcodes, ks, kz, vcodes, vs, vz, n, bits, kscheme, vscheme) = args
    L = n
    kc, kss, kzz = orc.unpack_cache(kcodes, ks, kz, [n], bits, 0, L)
    vc, vss, vzz = orc.unpack_cache(vcodes, vs, vz, [n], bits, 1, L)
    khat = orc.dequantize(kc, kss, kzz, [n], kscheme)
    vhat = orc.dequantize(vc, vss, vzz, [n], vscheme)
    q = orc.bf16_bits_to_f64(q_bits)
    orc.attend(q, khat, vhat, [n])
    _ = np


def oracle_pack_unit(args):
    """Packed inputs of one (sequence, kv head) unit, packed by the oracle from the
    workload's own pre-quantization values (runs in a pool worker)."""
    import numpy as np
    from oracle import kvq_oracle as orc
    w, seed, u = args
    lens = synth.seq_lens_for(w, seed)
    q = synth.query(w, seed)
    cs = synth.outlier_channels(w, seed)
    b, h = divmod(u, w.num_kv_heads)
    b %= w.batch
    n = int(lens[b])
    k = synth.kv_unit(w, seed, 0, b, h, n, "cpu", cs[h]).numpy()[None, None]
    v = synth.kv_unit(w, seed, 1, b, h, n, "cpu").numpy()[None, None]
    kcodes, ks, kz = orc.pack_cache(k, [n], w.bits, w.k_scheme, 0, group=w.group)
    vcodes, vs, vz = orc.pack_cache(v, [n], w.bits, w.v_scheme, 1, group=w.group)
    qb = q[b:b + 1, 4 * h:4 * h + 4].contiguous().view(torch.int16).numpy().view(np.uint16)
    return (qb, kcodes, ks, kz, vcodes, vs, vz, n, w.bits, w.k_scheme, w.v_scheme)


ORACLE_UNITS = 128  # default sample: about 10 core-seconds of oracle decode on the GPU host


class OracleTimer:
    """Times the CPU oracle on a bounded sample of the workload: the first
    `units` (sequence, kv head) units, packed once by the oracle (in the pool,
    untimed), then decoded (unpack + dequantize + attend, fp64) by one spawned
    process per host core."""

    def __init__(self, w, seed, units=None):
        import multiprocessing as mp
        total_units = w.batch * w.num_kv_heads
        self.units = min(units or ORACLE_UNITS, total_units)
        self.cores = max(1, min(host_cores(), self.units))
        lens = synth.seq_lens_for(w, seed)
        self.sample_lens = [int(lens[divmod(u, w.num_kv_heads)[0] % w.batch]) for u in range(self.units)]
        self.bytes = sum(((n + 127) // 128) * block_bytes_kv(w)
                         for n in self.sample_lens)
        self.sample = (f"{self.units} of {w.batch * w.num_kv_heads} (sequence, kv head) units "
                       f"({sum(self.sample_lens)} tokens), oracle unpack+dequantize+attend in fp64")
        old = os.environ.get("OMP_NUM_THREADS")
        os.environ["OMP_NUM_THREADS"] = "1"  # one core per worker
        self.pool = mp.get_context("spawn").Pool(self.cores)
        if old is None:
            os.environ.pop("OMP_NUM_THREADS", None)
        else:
            os.environ["OMP_NUM_THREADS"] = old
        self.jobs = self.pool.map(oracle_pack_unit, [(w, seed, u) for u in range(self.units)])
        self.pool.map(_oracle_unit, self.jobs[:self.cores])  # warm-up: imports and first touch

    def step(self) -> float:
        t0 = time.perf_counter()
        self.pool.map(_oracle_unit, self.jobs)
        return time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()


# ---------------------------------------------------------------- helpers
def host_cores() -> int:
    """Host cores this process may run on (its CPU affinity set)."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


def profile_traffic(workload: str, general: bool = False):
    """DRAM bytes per decode launch from the committed ncu record of the kernel
    that ran (`profiles/decode[_general]_<workload>_traffic.json`), if it was
    captured from the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"decode_{'general_' if general else ''}{workload}_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha256") != kernel_source_hash(general):
        return None
    return rec.get("dram_bytes_per_launch")


def kernel_source_hash(general: bool = False):
    """SHA-256 of the sources a decode kernel is compiled from, line comments
    and trailing blanks removed (a change of wording is not a new kernel)."""
    import re
    names = ("decode.cuh", "kvq_ptx.cuh", "kvq_internal.h")
    if general:
        names = ("decode_general.cuh", "decode_general.h") + names
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "bit_quantized_kv_decode_gb300", "csrc", name), encoding="utf-8") as f:
            text = f.read()
        code = "\n".join(line.rstrip() for line in re.sub(r"//[^\n]*", "", text).splitlines() if line.strip())
        h.update(code.encode("utf-8"))
    return h.hexdigest()


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist.get_rank(), world, int(os.environ.get("LOCAL_RANK", "0"))
    return 0, 1, 0


def max_over_ranks(x: float, world: int, dev) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------- main
def config_of(w):
    return {"workload": w.name, "batch": w.batch, "kv_heads": w.num_kv_heads, "q_heads": w.num_q_heads,
            "head_dim": w.head_dim, "seq_len": w.max_seq_len if w.ragged is None else f"log-uniform {w.ragged}",
            "bits": w.bits, "k_scheme": SCHEME_NAMES[w.k_scheme], "v_scheme": SCHEME_NAMES[w.v_scheme],
            "paged": w.paged, "group": w.group, "operands": "fp8 (E4M3 codes, 3-part E4M3 Q'/P')"}


def run_reference(args, w):
    rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return 0
    timer = OracleTimer(w, args.seed, args.oracle_units)
    for _ in range(min(args.warmup, 1)):
        timer.step()
    per_step = [timer.step() for _ in range(max(1, args.steps))]
    timer.close()
    ms = 1000.0 * sum(per_step) / len(per_step)
    value = timer.bytes / (ms / 1000.0) / 1e9
    line = {"impl": "reference", "metric": "effective KV-access HBM GB/s", "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": len(per_step), "warmup": min(args.warmup, 1), "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": timer.cores, "kind": "oracle",
                             "sample": timer.sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--seed", type=int, default=2024)
    ap.add_argument("--no-extra", action="store_true", help="skip the INT2 scheme sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-units", type=int, default=None)
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch (smaller cases for profiler captures)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--q-per-kv", type=int, choices=(1, 2, 4, 8), default=None,
                    help="query heads per KV head (the workloads use 4)")
    ap.add_argument("--k-scheme", choices=("token", "channel"), default=None,
                    help="override the workload's K quantization axis")
    ap.add_argument("--v-scheme", choices=("token", "channel"), default=None,
                    help="override the workload's V quantization axis")
    ap.add_argument("--operands", choices=("fp8", "bf16"), default="fp8",
                    help="tensor-core operand mode: fp8 (default) or the bf16 mode")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    w = synth.WORKLOADS[args.workload]
    if args.batch is not None:
        w = synth.shrink(w, batch=args.batch, name=f"{w.name}_b{args.batch}")
    if args.q_per_kv is not None and args.q_per_kv * w.num_kv_heads != w.num_q_heads:
        w = synth.shrink(w, num_q_heads=args.q_per_kv * w.num_kv_heads, name=f"{w.name}_g{args.q_per_kv}")
    for which, arg in (("k_scheme", args.k_scheme), ("v_scheme", args.v_scheme)):
        code = {v: k for k, v in SCHEME_NAMES.items()}.get(arg)
        if arg is not None and code != getattr(w, which):
            w = synth.shrink(w, **{which: code}, name=f"{w.name}_{which[0]}{arg[0]}")
    if args.impl == "reference":
        return run_reference(args, w)

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import bit_quantized_kv_decode_gb300 as kvq
    kvq.library()

    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    mode = 1 if args.operands == "bf16" else 0
    res = measure_kvq(w, args.seed + rank, args.steps, args.warmup, dev, e2e=not args.no_e2e, mode=mode)
    barrier(world)
    ms = max_over_ranks(res["ms"], world, dev)
    e2e_ms = max_over_ranks(res["e2e_ms"], world, dev) if "e2e_ms" in res else float("nan")
    extra = []
    if not args.no_extra and w.name == DEFAULT_WORKLOAD:
        w2 = synth.WORKLOADS["b128_l32k_int2"]
        for ks, vs in ((1, 0), (0, 0), (0, 1), (1, 1)):
            r2 = measure_kvq(w2, args.seed + rank, max(20, args.steps // 4), args.warmup, dev, ks, vs, e2e=False,
                             mode=mode)
            ms2 = max_over_ranks(r2["ms"], world, dev)
            extra.append({"workload": w2.name, "k_scheme": SCHEME_NAMES[ks], "v_scheme": SCHEME_NAMES[vs],
                          "ms_per_step": ms2, "GB/s": r2["bytes"] / (ms2 / 1e3) / 1e9,
                          "latency_us": ms2 * 1e3, "kernel": r2["kernel"]})
    e2m1 = []  # the 2-bit sweep again with the V codes placed as E2M1 in shared memory
    if not args.no_extra and w.name == DEFAULT_WORKLOAD and mode == 0:
        w2 = synth.WORKLOADS["b128_l32k_int2"]
        for ks, vs in ((1, 0), (0, 0), (0, 1), (1, 1)):
            r2 = measure_kvq(w2, args.seed + rank, 20, args.warmup, dev, ks, vs, e2e=False, flags=kvq.FLAG_E2M1_V)
            ms2 = max_over_ranks(r2["ms"], world, dev)
            e2m1.append({"workload": w2.name, "k_scheme": SCHEME_NAMES[ks], "v_scheme": SCHEME_NAMES[vs],
                         "v_operand": "E2M1 (code / 2) in shared memory", "ms_per_step": ms2,
                         "GB/s": r2["bytes"] / (ms2 / 1e3) / 1e9, "latency_us": ms2 * 1e3, "kernel": r2["kernel"]})
    configs = []
    if not args.no_extra and w.name == DEFAULT_WORKLOAD:
        for name in ("b8_l4k_int2", "paged_ragged_int2"):
            w3 = synth.WORKLOADS[name]
            r3 = measure_kvq(w3, args.seed + rank, max(20, args.steps // 4), args.warmup, dev, e2e=False, mode=mode)
            ms3 = max_over_ranks(r3["ms"], world, dev)
            lens3 = r3["lens"]
            configs.append({"workload": name, "k_scheme": SCHEME_NAMES[w3.k_scheme],
                            "v_scheme": SCHEME_NAMES[w3.v_scheme], "bits": w3.bits, "ms_per_step": ms3,
                            "GB/s": r3["bytes"] / (ms3 / 1e3) / 1e9, "latency_us": ms3 * 1e3,
                            "algorithmic_bytes": r3["bytes"], "l2": l2_note(r3),
                            "seq_lens": (f"{len(lens3)} sequences, min {min(lens3)}, max {max(lens3)}, "
                                         f"mean {sum(lens3) / len(lens3):.0f} tokens" if w3.ragged else
                                         f"{len(lens3)} x {lens3[0]} tokens"),
                            "paged": w3.paged, "kernel": r3["kernel"],
                            "split_kv": SPLIT_GENERAL if r3["general"] else SPLIT_SPECIALISED})
    geometry = []  # head dims 64 / 256 and groups of 32 / 64: the general-geometry kernel
    if not args.no_extra and w.name == DEFAULT_WORKLOAD:
        for name in ("b32_l32k_d256_g64_int4", "b32_l32k_d128_g32_int2", "b32_l32k_d64_g32_int2"):
            w4 = synth.WORKLOADS[name]
            r4 = measure_kvq(w4, args.seed + rank, 20, args.warmup, dev, e2e=False, mode=mode)
            ms4 = max_over_ranks(r4["ms"], world, dev)
            geometry.append({"workload": name, "head_dim": w4.head_dim, "group": w4.group, "bits": w4.bits,
                             "k_scheme": SCHEME_NAMES[w4.k_scheme], "v_scheme": SCHEME_NAMES[w4.v_scheme],
                             "ms_per_step": ms4, "GB/s": r4["bytes"] / (ms4 / 1e3) / 1e9, "latency_us": ms4 * 1e3,
                             "algorithmic_bytes": r4["bytes"], "l2": l2_note(r4), "operands": args.operands,
                             "kernel": r4["kernel"]})
    clk = clocks.summary(res["t0"], res["t1"])
    clocks.stop()
    if rank != 0:
        return 0
    peak, peak_kind = measured_peak()
    total_bytes = res["bytes"] * world
    value = total_bytes / (ms / 1e3) / 1e9
    achieved = res["bytes"] / (ms / 1e3) / 1e9
    for e in extra + configs + e2m1 + geometry:
        e["frac_of_peak"] = e["GB/s"] / peak
    line = {
        "metric": "effective KV-access HBM GB/s", "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "latency_us": ms * 1e3,
        "pct_of_peak": 100.0 * achieved / peak, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "data": "synthetic",
        "dtype": ("bf16 (tensor-core operands, fp32 accumulate)" if mode else
                  "fp8 (e4m3 tensor-core operands, fp32 accumulate)"),
        "config": dict(config_of(w), l2=l2_note(res),
                       **({"operands": "bf16 (exact BF16 codes, 2-part BF16 Q'/P')"} if mode else {})),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "kernel": res["kernel"],
                     "traffic": profile_traffic(w.name, res["general"]) if mode == 0 else None,
                     "algorithmic_bytes_per_launch": res["bytes"],
                     "duration_source": ("CUDA events around each kvq_decode_attn call (plan, decode and merge "
                                         "kernels)" if res["general"] else
                                         "CUDA events around each kvq_decode_attn call (counter memset + kernel)")},
        "e2e": ({"value": total_bytes / (e2e_ms / 1e3) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                 "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"]} if "e2e_ms" in res else None),
        "gpu_launches": res["launches"],
        "clocks": clk,
        "int2_sweep": extra,
        "int2_sweep_e2m1_v": e2m1,
        "other_configs": configs,
        "geometry_configs": geometry,
    }
    if not args.no_cpu_baseline and world == 1:
        timer = OracleTimer(w, args.seed, args.oracle_units)
        wall = min(timer.step() for _ in range(2))
        timer.close()
        line["cpu_baseline"] = {"value": timer.bytes / wall / 1e9, "unit": "GB/s", "cores": timer.cores,
                                "kind": "oracle", "sample": timer.sample, "wall_s": wall}
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
