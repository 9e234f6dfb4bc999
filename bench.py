#!/usr/bin/env python
"""Benchmark of one paged-KV attention step on GB300.

A step is the whole hot path on one synthetic batch: pa_cache_write (the new
tokens' K/V into their slots) then pa_forward (plan + split-KV attention, and
the multi-token path when the step has chunks).  The headline workload is the
Llama-3-8B single-layer decode shape (batch 256, 32 q / 8 kv heads, D=128,
bf16, lognormal contexts with median 1024, sigma 0.8, cap 8192); its KV
(~1.4 GB) is far larger than L2, so no flush is needed between steps.  The
mixed continuous-batching step (192 decodes + two 512-token chunks) is
reported alongside as tokens/s per layer.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line.  `--impl reference` times the fp64 CPU oracle on a
bounded sample of the same workload instead (there is no other reference
implementation of this path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode paged-attn HBM GB/s & % of GB300 peak; mixed-step tokens/s per layer"
HEADLINE = "llama3_8b_decode"
MIXED = "mixed_step"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# nominal GB300 figures (context beside the measured peaks): HBM3e 7.9 TB/s,
# dense bf16 tensor 2.25 PFLOP/s
NOMINAL_HBM_GBS = 7900.0
NOMINAL_BF16_TFLOPS = 2250.0
WORKLOAD_TEXT = {
    "llama3_8b_decode": "Llama-3-8B single-layer decode: batch 256, 32 q / 8 kv heads, head_size 128, "
                        "bf16, context lognormal(median 1024, sigma 0.8, cap 8192), block_size 16, "
                        "random block tables, pool 1.2x needed",
    "mixed_step": "mixed step, Llama-3-8B heads, bf16: 192 decodes (context U[256,4096]) + 2 chunked "
                  "prefills of 512 (prior 0 and 1536), 1216 tokens, half the decodes share 64 prefix blocks",
}


# ---------------------------------------------------------------------------
# Algorithmic work of a step (counted from the inputs, never from kernels)
# ---------------------------------------------------------------------------

def step_work(spec, meta) -> dict:
    """Bytes the method must move and prefill flops, from the step's metadata.

    decode_bytes: unique KV slots read by q_len==1 requests (a shared prefix
    block counted once) x Hkv x D x 2 (K,V) x e, plus their q and out rows,
    block-table entries, seq_lens and query_start_loc.
    write_bytes: new k,v read + written into the cache, plus slot_mapping.
    chunk_bytes/flops: the same for q_len>1 requests; flops = 4 x D x Hq x
    (visible (query, key) pairs)."""
    import numpy as np
    e = 2 if spec.dtype == "bf16" else 4
    Hq, Hkv, D, bs = spec.num_q_heads, spec.num_kv_heads, spec.head_size, spec.block_size
    bt = meta.block_tables
    dec_slots, chk_slots = [], []
    table_dec = table_chk = 0
    pairs = 0
    for r in range(spec.num_seqs):
        S, L = int(spec.seq_lens[r]), int(spec.q_lens[r])
        p = np.arange(S)
        slots = bt[r, p // bs].astype(np.int64) * bs + p % bs
        nb = -(-S // bs)
        if L == 1:
            dec_slots.append(slots)
            table_dec += nb
        else:
            chk_slots.append(slots)
            table_chk += nb
            pairs += sum(S - L + j + 1 for j in range(L))
    row = Hkv * D * e
    n_dec = sum(1 for L in spec.q_lens if L == 1)
    n_chk_tok = int(sum(L for L in spec.q_lens if L > 1))
    uniq = lambda lst: int(len(np.unique(np.concatenate(lst)))) if lst else 0  # noqa: E731
    meta_bytes = 4 * (2 * spec.num_seqs + 1)
    kv_bytes = uniq(dec_slots) * row * 2
    decode_bytes = (kv_bytes + 2 * n_dec * Hq * D * e + 4 * table_dec + meta_bytes)
    chunk_bytes = (uniq(chk_slots) * row * 2 + 2 * n_chk_tok * Hq * D * e + 4 * table_chk)
    T = spec.num_tokens
    write_bytes = 2 * 2 * T * row + 8 * T
    return dict(decode_bytes=decode_bytes, kv_bytes=kv_bytes, chunk_bytes=chunk_bytes,
                write_bytes=write_bytes,
                step_bytes=decode_bytes + chunk_bytes + write_bytes,
                chunk_flops=4.0 * D * Hq * pairs, tokens=T)


def measured_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops() -> tuple[float, str]:
    """Dense bf16 peak (burst) from MEASURED_PEAKS.json, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in ("pa_attn_mma.cuh", "pa_attn_mma_bf16.cu", "pa_device.cuh"):
        with open(os.path.join(ROOT, "paged_kv_attention_04_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the decode kernel from the committed ncu summary
    (profiles/traffic.txt), if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if parts and not parts[0].startswith("#") and parts[0] == workload:
                    if parts[1] == kernel_source_hash():
                        return float(parts[2])
    except OSError:
        pass
    return None


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid: str | None):
        self.samples = []
        self.proc = None
        self.uuid = gpu_uuid
        self.marks = {}

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, name):
        self.marks[name] = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.45)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        t0, t1 = self.marks.get("timed_start", 0), self.marks.get("timed_end", 1e30)
        rows = [s for t, s in self.samples if t0 - 0.25 <= t <= t1 + 0.25]
        window = "timed"
        if not rows:
            w0 = self.marks.get("warm_start", 0)
            rows = [s for t, s in self.samples if w0 <= t <= t1 + 0.3]
            window = "warmup+timed"
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in rows:
            parts = [p.strip() for p in s.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "window": window}


# ---------------------------------------------------------------------------
# CPU oracle timing (runs in a child process with single-threaded BLAS)
# ---------------------------------------------------------------------------

def oracle_worker(name: str, min_seconds: float, stride: int, steps: int, warmup: int,
                  step_budget: float, offset: int = 0, sync: bool = False) -> None:
    """Time the fp64 oracle on a sample of workload `name`: every `stride`-th
    request from `offset` (stride 0: chosen so one pass fits `step_budget` seconds), each
    with a private copy of its blocks; one pass = slot write + attention of the
    sampled requests.  With steps > 0, times warmup + steps passes and reports
    the timed ones; else repeats passes until min_seconds.  With sync, prints
    "ready" once the sample is prepared and starts timing when a line arrives
    on stdin (so that concurrent workers time the same interval).  Prints JSON."""
    import numpy as np

    import oracle
    from paged_kv_attention_04_gb300 import workloads as W
    spec = W.CONFIGS[name]()
    st = W.make_step(spec)
    b = W.to_numpy_bits
    bt = st.block_tables.numpy()
    qsl = st.query_start_loc.numpy()
    scale = 1.0 / np.sqrt(spec.head_size)

    def prep(r):
        S, L = int(spec.seq_lens[r]), int(spec.q_lens[r])
        nb = -(-S // 16)
        blocks = bt[r, :nb].astype(np.int64)
        t0, t1 = int(qsl[r]), int(qsl[r + 1])
        pos = np.arange(S - L, S)
        return dict(kc=b(st.k_cache[blocks]), vc=b(st.v_cache[blocks]), q=b(st.q[t0:t1]),
                    k=b(st.k[t0:t1]), v=b(st.v[t0:t1]), slots=(pos // 16) * 16 + pos % 16,
                    S=S, L=L, nb=nb)

    def run(samples):
        for s in samples:
            kc, vc = oracle.cache_write(s["k"], s["v"], s["slots"], s["kc"], s["vc"])
            oracle.paged_attention(s["q"], kc, vc, np.arange(s["nb"])[None, :], np.array([s["S"]]),
                                   np.array([0, s["L"]]), scale, spec.num_kv_heads)

    if stride <= 0:
        probe = [prep(r) for r in range(0, spec.num_seqs, 32)]
        t = time.perf_counter()
        run(probe)
        per_req = (time.perf_counter() - t) / len(probe)
        n = int(max(1, min(spec.num_seqs, step_budget / max(per_req, 1e-6))))
        stride = max(1, spec.num_seqs // n)
    reqs = list(range(offset, spec.num_seqs, stride))
    samples = [prep(r) for r in reqs]
    sub = W.custom_spec("sample", spec.dtype, spec.num_q_heads, spec.num_kv_heads, spec.head_size,
                        [s["L"] for s in samples], [s["S"] for s in samples])
    work = step_work(sub, W.make_meta(sub))
    del st
    if sync:
        print("ready", flush=True)
        sys.stdin.readline()
    times = []
    if steps > 0:
        for i in range(warmup + steps):
            t = time.perf_counter()
            run(samples)
            if i >= warmup:
                times.append(time.perf_counter() - t)
    else:
        elapsed = 0.0
        while elapsed < min_seconds or not times:
            t = time.perf_counter()
            run(samples)
            times.append(time.perf_counter() - t)
            elapsed += times[-1]
    print(json.dumps({"seconds": sum(times), "reps": len(times), "requests": len(reqs),
                      "stride": stride, "bytes_per_rep": work["step_bytes"],
                      "tokens_per_rep": work["tokens"]}))


def _oracle_cmd_env(name, min_seconds, stride, steps, warmup, step_budget, offset=0, sync=False):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-worker", name,
           "--oracle-seconds", str(min_seconds), "--oracle-stride", str(stride),
           "--oracle-offset", str(offset),
           *(["--oracle-sync"] if sync else []),
           "--steps", str(steps), "--warmup", str(warmup), "--oracle-budget", str(step_budget)]
    return cmd, env


def time_oracle(name: str, min_seconds: float = 10.0, stride: int = 1, steps: int = 0,
                warmup: int = 0, step_budget: float = 1.0) -> dict:
    cmd, env = _oracle_cmd_env(name, min_seconds, stride, steps, warmup, step_budget)
    res = subprocess.run(cmd, capture_output=True, text=True, env=env, cwd=ROOT)
    if res.returncode != 0:
        raise RuntimeError(f"oracle worker failed: {res.stderr[-2000:]}")
    return json.loads(res.stdout.strip().splitlines()[-1])


def time_oracle_all_cores(name: str, min_seconds: float = 10.0) -> dict:
    """The same single-threaded oracle in one process per host core, each on a
    disjoint share of the requests (every n-th from its own offset), all at
    once: every worker prepares its sample, then all start timing together.
    Returns the summed bytes per second, the cores used and the requests."""
    from paged_kv_attention_04_gb300 import workloads as W
    n_req = W.CONFIGS[name]().num_seqs
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    n = max(1, min(n or 1, n_req))
    procs = []
    for j in range(n):
        cmd, env = _oracle_cmd_env(name, min_seconds, n, 0, 0, 1.0, offset=j, sync=True)
        procs.append(subprocess.Popen(cmd, stdin=subprocess.PIPE, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True, env=env, cwd=ROOT))
    try:
        for pr in procs:
            if pr.stdout.readline().strip() != "ready":
                raise RuntimeError(f"oracle worker failed: {pr.stderr.read()[-2000:]}")
        for pr in procs:
            pr.stdin.write("go\n")
            pr.stdin.flush()
        gbs, reqs, secs = 0.0, 0, []
        for pr in procs:
            out, err = pr.communicate()
            if pr.returncode != 0:
                raise RuntimeError(f"oracle worker failed: {err[-2000:]}")
            o = json.loads(out.strip().splitlines()[-1])
            gbs += o["bytes_per_rep"] * o["reps"] / o["seconds"] / 1e9
            reqs += o["requests"]
            secs.append(o["seconds"])
    finally:
        for pr in procs:
            if pr.poll() is None:
                pr.kill()
                pr.wait()
    return {"gbs": gbs, "cores": n, "requests": reqs, "seconds": min(secs)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(local)
    return world, rank, local


def dist_max(x: float, world: int) -> float:
    """Maximum of x over all ranks (x itself on one rank).  Uses the process
    group's backend: CUDA tensors under nccl, CPU tensors under gloo."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(bytes_per_rank: float, ms_max: float, world: int) -> float:
    """Whole-job GB/s for `world` replicas that each moved bytes_per_rank, timed
    by the slowest rank."""
    return world * bytes_per_rank / (ms_max * 1e-3) / 1e9


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class StepRunner:
    """Device-resident step of one workload through the C ABI."""

    def __init__(self, name: str, seed_offset: int = 0, fp8_scales: tuple | None = None,
                 requests: slice | None = None):
        import torch

        import paged_kv_attention_04_gb300 as P
        from paged_kv_attention_04_gb300 import workloads as W
        self.P, self.torch = P, torch
        fn = W.CONFIGS[name]
        spec = fn()
        if seed_offset:
            spec.seed += seed_offset
        if requests is not None:  # a subset of the workload's requests
            spec.seq_lens = spec.seq_lens[requests]
            spec.q_lens = spec.q_lens[requests]
            if spec.sharing is not None:
                spec.sharing = spec.sharing[requests]
        self.spec = spec
        self.meta = W.make_meta(spec)
        self.st = W.make_step(spec, device="cuda")
        st = self.st
        if fp8_scales:
            # 8-bit cache: the bf16 history pool as E4M3 codes of x / scale
            ks, vs = fp8_scales
            st.k_cache = (st.k_cache.float() / ks).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
            st.v_cache = (st.v_cache.float() / vs).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
            self.layout = P.layout_of(st.k_cache, spec.num_q_heads, k_scale=ks, v_scale=vs)
        else:
            self.layout = P.layout_of(st.k_cache, spec.num_q_heads)
        self.ws = P.alloc_workspace(self.layout, spec.num_seqs, spec.num_tokens, st.max_seq_len)
        self.out = torch.empty_like(st.q)
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.work = step_work(spec, self.meta)
        self.launches_per_step = 3 + (1 if st.max_query_len > 1 else 0)

    def step(self, q=None, k=None, v=None, slots=None, bt=None, sl=None, qsl=None):
        st, P = self.st, self.P
        q = st.q if q is None else q
        P.pa_cache_write(st.k if k is None else k, st.v if v is None else v,
                         st.slot_mapping if slots is None else slots, st.k_cache, st.v_cache,
                         self.layout, self.status)
        P.pa_forward(q, st.k_cache, st.v_cache, st.block_tables if bt is None else bt,
                     st.seq_lens if sl is None else sl, st.query_start_loc if qsl is None else qsl,
                     st.max_query_len, st.max_seq_len, st.scale, self.out, self.ws, self.layout,
                     self.status)

    FLUSH_TEXT = ("flushed before every step, outside the timed events: a 256 MiB buffer "
                  "(twice L2) written, then read back, so the step starts with none of its "
                  "inputs in L2 and no dirty lines left to write back")

    def flush_l2(self):
        """Write 256 MiB (twice the L2), then read it, so the next step starts
        with a cold L2: the read evicts the written lines, whose write-back to
        HBM would otherwise land inside the timed step."""
        if not hasattr(self, "_flush"):
            self._flush = self.torch.empty(256 << 20, dtype=self.torch.uint8, device="cuda")
        self._flush.zero_()
        self._flush.view(self.torch.int32).sum()

    def time_device(self, steps: int, warmup: int, world: int, clocks: ClockSampler | None = None,
                    flush: bool = False, serial_kernels: bool = False):
        """Inputs resident in HBM; returns (ms per step, decode-kernel ms per launch,
        prefill-kernel ms per launch or None), the kernel times being means over
        the launches (the event clock ticks in ~2 us steps; a launch starts at a
        random phase of the tick, so the mean of many launches resolves what
        one reading, or a median of them, rounds away).  The steps are timed in
        one loop with no events inside a step; the kernels are timed in a second
        loop with events around each (events between the plan and the decode
        kernel would cost the step their launch overlap).  With flush, L2 is
        flushed before every step, outside the timed events."""
        torch, P = self.torch, self.P
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize()
        has_prefill = self.st.max_query_len >= 16 and self.spec.dtype == "bf16"

        def loop(kernel_events):
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(steps)]
            pevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for _ in range(steps)]
            steps_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                        for _ in range(steps if flush else 1)]
            barrier(world)
            torch.cuda.synchronize()
            if not flush:
                steps_ev[0][0].record()
            for i in range(steps):
                if flush:
                    self.flush_l2()
                    steps_ev[i][0].record()
                if kernel_events:
                    P.pa_set_profile_events(evs[i][0], evs[i][1])
                    if has_prefill:
                        P.pa_set_prefill_profile_events(pevs[i][0], pevs[i][1])
                self.step()
                if flush:
                    steps_ev[i][1].record()
            if not flush:
                steps_ev[0][1].record()
            torch.cuda.synchronize()
            barrier(world)
            P.pa_set_profile_events(None, None)
            P.pa_set_prefill_profile_events(None, None)
            if kernel_events:
                dec = statistics.fmean(a.elapsed_time(b) for a, b in evs)
                pf = statistics.fmean(a.elapsed_time(b) for a, b in pevs) if has_prefill else None
                return dec, pf
            return sum(a.elapsed_time(b) for a, b in steps_ev) / steps

        if clocks:
            clocks.mark("timed_start")
        step_ms = loop(False)
        if clocks:
            clocks.mark("timed_end")
        if serial_kernels and has_prefill:
            # the prefill kernel on the caller's stream: its events then time it
            # alone, not also the wait for SMs that the decode kernel's CTAs
            # (resident early, with no work in a prefill-only step) hold
            P.pa_set_prefill_overlap(False)
        try:
            dec_ms, pf_ms = loop(True)
        finally:
            P.pa_set_prefill_overlap(True)
        return step_ms, dec_ms, pf_ms

    def time_graph(self, steps: int, warmup: int, world: int, flush: bool = False) -> float:
        """The same step captured once in a CUDA graph and replayed; ms per step
        (with flush, L2 is flushed before every replay, outside the timed events)."""
        torch = self.torch
        self.step()  # per-device set-up happens on an eager call, before capture
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g):
                self.step()
        torch.cuda.current_stream().wait_stream(s)
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        barrier(world)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps if flush else 1)]
        if not flush:
            evs[0][0].record()
        for i in range(steps):
            if flush:
                self.flush_l2()
                evs[i][0].record()
            g.replay()
            if flush:
                evs[i][1].record()
        if not flush:
            evs[0][1].record()
        torch.cuda.synchronize()
        barrier(world)
        del g
        return sum(a.elapsed_time(b) for a, b in evs) / steps

    def time_e2e(self, steps: int, warmup: int, world: int):
        """Same step with this step's inputs copied from pinned host memory
        and the output copied back, inside the timed region.  The inputs sit
        in one pinned staging buffer (each at a 256-byte offset) and go over
        in one copy, as a serving loop would stage a step's metadata."""
        torch = self.torch
        st = self.st
        names = ("q", "k", "v", "slot_mapping", "block_tables", "seq_lens", "query_start_loc")
        srcs = {n: getattr(st, n) for n in names}
        offs, off = {}, 0
        for n in names:
            offs[n] = off
            off = (off + srcs[n].numel() * srcs[n].element_size() + 255) // 256 * 256
        host_buf = torch.zeros(off, dtype=torch.uint8).pin_memory()
        dev_buf = torch.empty(off, dtype=torch.uint8, device=self.out.device)

        def view(buf, n):
            t = srcs[n]
            nb = t.numel() * t.element_size()
            return buf[offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)

        for n in names:
            view(host_buf, n).copy_(srcs[n].cpu())
        dev = {n: view(dev_buf, n) for n in names}
        out_host = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        h2d = off
        d2h = out_host.numel() * out_host.element_size()

        def one():
            dev_buf.copy_(host_buf, non_blocking=True)
            self.step(q=dev["q"], k=dev["k"], v=dev["v"], slots=dev["slot_mapping"],
                      bt=dev["block_tables"], sl=dev["seq_lens"], qsl=dev["query_start_loc"])
            out_host.copy_(self.out, non_blocking=True)

        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            one()
        e1.record()
        torch.cuda.synchronize()
        barrier(world)
        return e0.elapsed_time(e1) / steps, h2d, d2h


def _check_status(runner, what: str) -> None:
    if int(runner.status.item()) != 0:
        raise RuntimeError(f"{what}: device status {int(runner.status.item())}")


def run_gpu_arm(args):
    import torch

    import paged_kv_attention_04_gb300 as P
    from paged_kv_attention_04_gb300 import build
    build.build()
    world, rank, local = dist_setup()
    if world != args.gpus:
        print(f"warning: WORLD_SIZE={world} but --gpus {args.gpus}", file=sys.stderr)
    dev_uuid = None
    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        dev_uuid = u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    seed_off = rank * 1000 if world > 1 else 0
    peak, peak_src = measured_peaks()
    bf16_peak = measured_bf16_tflops()
    half = max(3, args.steps // 2)

    # ---- headline: Llama-3-8B decode step
    runner = StepRunner(HEADLINE, seed_offset=seed_off)
    clocks = ClockSampler(dev_uuid)
    clocks.start()
    time.sleep(0.3)
    clocks.mark("warm_start")
    ms, dec_ms, _ = runner.time_device(args.steps, args.warmup, world, clocks)
    clock_info = clocks.stop()
    _check_status(runner, "headline")
    ms_max = dist_max(ms, world)
    dec_max = dist_max(dec_ms, world)
    w = runner.work
    value = replica_value(w["step_bytes"], ms_max, world)
    graph_ms = dist_max(runner.time_graph(args.steps, args.warmup, world), world)
    e2e_ms, h2d, d2h = runner.time_e2e(max(3, args.steps // 4), max(3, args.warmup), world)
    e2e_ms = dist_max(e2e_ms, world)
    e2e_value = replica_value(w["step_bytes"], e2e_ms, world)
    achieved = w["decode_bytes"] / (dec_max * 1e-3) / 1e9
    traffic = recorded_traffic(HEADLINE)
    launches = runner.launches_per_step * args.steps
    del runner
    torch.cuda.empty_cache()

    # ---- mixed continuous-batching step: prefill overlapped with decode, and serial
    mixed = StepRunner(MIXED, seed_offset=seed_off)
    mms, mdec, _ = (dist_max(x, world) if x is not None else None
                    for x in mixed.time_device(half, args.warmup, world))
    mgraph = dist_max(mixed.time_graph(half, args.warmup, world), world)
    P.pa_set_prefill_overlap(False)
    try:
        sms_, sdec, spf = (dist_max(x, world) for x in mixed.time_device(half, args.warmup, world))
    finally:
        P.pa_set_prefill_overlap(True)
    _check_status(mixed, "mixed step")
    mw = mixed.work
    del mixed
    torch.cuda.empty_cache()
    # the step's decode requests alone: the decode kernel's standalone rate
    md = StepRunner(MIXED, seed_offset=seed_off, requests=slice(0, -2))
    _, adec, _ = md.time_device(half, args.warmup, world)
    adec = dist_max(adec, world)
    _check_status(md, "mixed-step decodes alone")
    del md
    torch.cuda.empty_cache()
    mixed_info = {
        "workload": WORKLOAD_TEXT[MIXED],
        "tokens_per_s_per_layer": world * mw["tokens"] / (mms * 1e-3),
        "ms_per_step": mms,
        "serial_ms_per_step": sms_,
        "overlap_speedup": sms_ / mms,
        "graph_ms_per_step": mgraph,
        "decode_kernel_ms": mdec,
        "decode_gbs": mw["decode_bytes"] / (mdec * 1e-3) / 1e9,
        "serial_decode_kernel_ms": sdec,
        "serial_prefill_kernel_ms": spf,
        "serial_prefill_tflops": mw["chunk_flops"] / (spf * 1e-3) / 1e12,
        "decode_alone_kernel_ms": adec,
        "decode_alone_gbs": mw["decode_bytes"] / (adec * 1e-3) / 1e9,
        "decode_in_step_vs_alone": adec / mdec,
        "timed": "ms_per_step: pa_cache_write + pa_forward back to back with no events inside a "
                 "step (prefill kernel on the library side stream beside the decode kernel); "
                 "serial_ms_per_step: the same with pa_set_prefill_overlap(0) (prefill kernel "
                 "on the caller's stream before the decode kernel); kernel times: means of "
                 "events around each kernel in a second loop (overlapped, the prefill kernel's "
                 "stop event waits for CTAs that only start when decode CTAs leave, so only the "
                 "serial prefill time is reported); decode_alone: the 192 decode requests as a "
                 "step of their own",
    }

    # ---- the mixed step over an 8-bit (E4M3) KV cache
    mf = StepRunner(MIXED, seed_offset=seed_off, fp8_scales=(0.01, 0.01))
    fms_, fmdec, _ = mf.time_device(half, args.warmup, world)
    fms_, fmdec = dist_max(fms_, world), dist_max(fmdec, world)
    _check_status(mf, "mixed step, fp8")
    fmw = mf.work
    mixed_info["fp8_kv"] = {
        "ms_per_step": fms_,
        "tokens_per_s_per_layer": world * fmw["tokens"] / (fms_ * 1e-3),
        "decode_kernel_ms": fmdec,
        "decode_gbs": (fmw["decode_bytes"] - fmw["kv_bytes"] // 2) / (fmdec * 1e-3) / 1e9,
        "note": "KV cache E4M3 (scales 0.01): decode reads 8-bit codes, the chunks run on "
                "the tensor-core prefill kernel over codes widened to f16 in shared memory",
    }
    del mf
    torch.cuda.empty_cache()

    # ---- the mixed step's two prefill chunks alone: the tensor-core kernel's own rate
    pf = StepRunner(MIXED, seed_offset=seed_off, requests=slice(-2, None))
    pms, _, ppf = pf.time_device(half, args.warmup, world, flush=True, serial_kernels=True)
    pms, ppf = dist_max(pms, world), dist_max(ppf, world)
    _check_status(pf, "prefill chunks")
    pf_tflops = pf.work["chunk_flops"] / (ppf * 1e-3) / 1e12
    prefill_info = {
        "workload": "the mixed step's two chunked prefills alone: 512 tokens at prior 0 and "
                    "512 at prior 1536, Llama-3-8B heads, bf16",
        "ms_per_step": pms,
        "prefill_kernel_ms": ppf,
        "tflops": pf_tflops,
        "frac_of_bf16_peak": pf_tflops / bf16_peak[0],
        "frac_of_nominal_bf16": pf_tflops / NOMINAL_BF16_TFLOPS,
        "step_tflops": pf.work["chunk_flops"] / (pms * 1e-3) / 1e12,
        "peak_tflops": bf16_peak[0], "peak_source": bf16_peak[1],
        "flops": pf.work["chunk_flops"],
        "timed": "tflops: flops / mean event time of the tensor-core prefill kernel, timed "
                 "in a second loop with the prefill kernel on the caller's stream; "
                 "ms_per_step: pa_cache_write + pa_forward (plan, prefill kernel; default "
                 "side-stream schedule); L2 "
                 + StepRunner.FLUSH_TEXT + "; flops = 4 x D x Hq x visible (query, key) pairs",
    }
    del pf
    torch.cuda.empty_cache()

    # ---- one long chunk: the tensor-core kernel in its steady state (56 KV tiles a unit)
    pl = StepRunner("long_prefill_chunk", seed_offset=seed_off)
    lms, _, lpf = pl.time_device(half, args.warmup, world, flush=True, serial_kernels=True)
    lms, lpf = dist_max(lms, world), dist_max(lpf, world)
    _check_status(pl, "long prefill")
    pl_tflops = pl.work["chunk_flops"] / (lpf * 1e-3) / 1e12
    prefill_long_info = {
        "workload": "one 2048-token prefill chunk at prior context 6144 (rows see up to 8192 "
                    "keys), Llama-3-8B heads, bf16",
        "ms_per_step": lms,
        "prefill_kernel_ms": lpf,
        "tflops": pl_tflops,
        "frac_of_bf16_peak": pl_tflops / bf16_peak[0],
        "frac_of_nominal_bf16": pl_tflops / NOMINAL_BF16_TFLOPS,
        "step_tflops": pl.work["chunk_flops"] / (lms * 1e-3) / 1e12,
        "peak_tflops": bf16_peak[0], "peak_source": bf16_peak[1],
        "flops": pl.work["chunk_flops"],
        "timed": "as prefill_chunks",
    }
    del pl
    torch.cuda.empty_cache()
    plf = StepRunner("long_prefill_chunk", seed_offset=seed_off, fp8_scales=(0.01, 0.01))
    lfms, _, lfpf = plf.time_device(half, args.warmup, world, flush=True, serial_kernels=True)
    lfms, lfpf = dist_max(lfms, world), dist_max(lfpf, world)
    _check_status(plf, "long prefill, fp8")
    prefill_long_info["fp8_kv"] = {
        "ms_per_step": lfms,
        "prefill_kernel_ms": lfpf,
        "tflops": plf.work["chunk_flops"] / (lfpf * 1e-3) / 1e12,
        "frac_of_bf16_peak": plf.work["chunk_flops"] / (lfpf * 1e-3) / 1e12 / bf16_peak[0],
        "kernel": "the tensor-core prefill kernel over E4M3 codes staged by TMA and widened to "
                  "f16 in shared memory (f16 products)",
    }
    del plf
    torch.cuda.empty_cache()

    # ---- short chunks after long prompts: prefill units split over their KV
    lp = StepRunner("long_prior_chunks", seed_offset=seed_off)
    pps, _, ppk = lp.time_device(half, args.warmup, world, flush=True, serial_kernels=True)
    pps, ppk = dist_max(pps, world), dist_max(ppk, world)
    _check_status(lp, "long-prior chunks")
    lpw = lp.work
    long_prior_info = {
        "workload": "short prefill chunks late in long prompts: 64 tokens after 32768 and 16 "
                    "after 98304, Llama-3-8B heads, bf16",
        "ms_per_step": pps,
        "prefill_kernel_ms": ppk,
        "kv_gbs": lpw["chunk_bytes"] / (ppk * 1e-3) / 1e9,
        "frac_of_hbm_peak": lpw["chunk_bytes"] / (ppk * 1e-3) / 1e9 / peak,
        "tflops": lpw["chunk_flops"] / (ppk * 1e-3) / 1e12,
        "bound": "hbm: each query tile reads all its prior KV once (bytes = unique KV slots "
                 "read + q + out + block tables)",
        "algorithmic_bytes": lpw["chunk_bytes"], "flops": lpw["chunk_flops"],
        "l2": StepRunner.FLUSH_TEXT,
        "timed": "prefill kernel: mean event time in a second loop with the prefill kernel on "
                 "the caller's stream",
    }
    del lp
    torch.cuda.empty_cache()

    # ---- long-context decode: 16 requests of 32K-128K tokens, split-KV + merge
    lc = StepRunner("long_context_decode", seed_offset=seed_off)
    cms, cdec, _ = lc.time_device(half, args.warmup, world)
    cms, cdec = dist_max(cms, world), dist_max(cdec, world)
    _check_status(lc, "long-context decode")
    lw = lc.work
    long_info = {
        "workload": "long-context decode: batch 16, context U[32768,131072], 32 q / 8 kv heads, "
                    "D=128, bf16, random block tables over a 9 GB pool",
        "ms_per_step": cms,
        "decode_kernel_ms": cdec,
        "decode_gbs": lw["decode_bytes"] / (cdec * 1e-3) / 1e9,
        "decode_frac_of_peak": lw["decode_bytes"] / (cdec * 1e-3) / 1e9 / peak,
        "step_gbs": world * lw["step_bytes"] / (cms * 1e-3) / 1e9,
        "algorithmic_bytes_per_launch": lw["decode_bytes"],
        "l2": "no flush: KV read per step (5.8 GB) > L2",
    }
    del lc
    torch.cuda.empty_cache()

    # ---- the headline shape over an 8-bit (E4M3) KV cache: half the KV bytes per token
    f8 = StepRunner(HEADLINE, seed_offset=seed_off, fp8_scales=(0.01, 0.01))
    fms, fdec, _ = f8.time_device(args.steps, args.warmup, world)
    fms, fdec = dist_max(fms, world), dist_max(fdec, world)
    _check_status(f8, "fp8 decode")
    fkv = f8.work["decode_bytes"] - f8.work["kv_bytes"] // 2  # KV counted at 1 byte/element
    fp8_info = {
        "workload": WORKLOAD_TEXT[HEADLINE] + ", KV cache FP8 E4M3 (per-tensor scales)",
        "ms_per_step": fms, "decode_kernel_ms": fdec,
        "decode_gbs": fkv / (fdec * 1e-3) / 1e9,
        "decode_frac_of_peak": fkv / (fdec * 1e-3) / 1e9 / peak,
        "tokens_per_s": world * f8.spec.num_tokens / (fms * 1e-3),
    }
    del f8
    torch.cuda.empty_cache()

    # ---- a small decode step (79 MB of KV) where launch overhead is visible
    small = StepRunner("tinyllama_decode", seed_offset=seed_off)
    sms, sdec, _ = small.time_device(args.steps, args.warmup, world, flush=True)
    sms, sdec = dist_max(sms, world), dist_max(sdec, world)
    sgraph = dist_max(small.time_graph(args.steps, args.warmup, world, flush=True), world)
    _check_status(small, "tinyllama decode")
    sw = small.work
    small_info = {
        "workload": "TinyLlama-1.1B single-layer decode: batch 64, 32 q / 4 kv heads, D=64, bf16, "
                    "context U[128,2048]",
        "ms_per_step": sms, "graph_ms_per_step": sgraph, "decode_kernel_ms": sdec,
        "decode_gbs": sw["decode_bytes"] / (sdec * 1e-3) / 1e9,
        "decode_frac_of_peak": sw["decode_bytes"] / (sdec * 1e-3) / 1e9 / peak,
        "graph_step_gbs": world * sw["step_bytes"] / (sgraph * 1e-3) / 1e9,
        "l2": StepRunner.FLUSH_TEXT,
    }
    del small
    torch.cuda.empty_cache()

    # ---- the tiny fp32 decode step: 4 requests, latency-bound
    tiny = StepRunner("tiny_decode_f32", seed_offset=seed_off)
    tms, tdec, _ = tiny.time_device(args.steps, args.warmup, world, flush=True)
    tms, tdec = dist_max(tms, world), dist_max(tdec, world)
    tgraph = dist_max(tiny.time_graph(args.steps, args.warmup, world, flush=True), world)
    _check_status(tiny, "tiny fp32 decode")
    tiny_info = {
        "workload": "tiny fp32 decode: 4 requests, seq_lens {1,17,33,64}, 4 q / 2 kv heads, "
                    "D=64, 32-block pool",
        "us_per_step": tms * 1e3, "graph_us_per_step": tgraph * 1e3,
        "decode_kernel_us": tdec * 1e3,
        "decode_bytes": tiny.work["decode_bytes"],
        "l2": StepRunner.FLUSH_TEXT,
    }
    del tiny
    torch.cuda.empty_cache()

    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[HEADLINE], "step": "pa_cache_write + pa_forward",
                   "l2": "no flush: KV read per step (1.4 GB) > L2 (126 MB)",
                   "parallelism": f"{world} replicas" if world > 1 else "single GPU",
                   "algorithmic_bytes_per_step": w["step_bytes"]},
        "roofline": {"bound": "hbm",
                     "kernel": "attn_mma_kernel<128,4,1,4,2,0,0> (decode, query rows as M)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_src, "traffic": traffic,
                     "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": w["decode_bytes"], "kernel_ms": dec_max},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "graph_ms_per_step": graph_ms,
        "gpu_launches": launches,
        "clocks": clock_info,
        "mixed": mixed_info,
        "long_context_decode": long_info,
        "tiny_decode_f32": tiny_info,
        "tinyllama_decode": small_info,
        "fp8_kv": fp8_info,
        "prefill_chunks": prefill_info,
        "prefill_long": prefill_long_info,
        "long_prior_chunks": long_prior_info,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        o = time_oracle(HEADLINE, min_seconds=args.oracle_seconds, stride=args.oracle_stride)
        line["cpu_baseline"] = {
            "value": o["bytes_per_rep"] * o["reps"] / o["seconds"] / 1e9, "unit": "GB/s",
            "cores": 1, "kind": "oracle",
            "sample": f"{o['requests']} of 256 requests (every {o['stride']}th), each with its own "
                      f"blocks: fp64 slot write + attention, {o['reps']} passes, "
                      f"{o['seconds']:.1f} s on 1 core"}
        a = time_oracle_all_cores(HEADLINE, min_seconds=args.oracle_seconds)
        line["cpu_baseline_all_cores"] = {
            "value": a["gbs"], "unit": "GB/s", "cores": a["cores"], "kind": "oracle",
            "sample": f"all 256 requests split over {a['cores']} single-threaded processes "
                      f"(every {a['cores']}th request each, {a['requests']} in all), timed "
                      f"together for at least {a['seconds']:.1f} s"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    # each step is one oracle pass over a sample sized so the run takes ~2 minutes
    budget = 120.0 / max(1, args.steps + args.warmup)
    o = time_oracle(HEADLINE, stride=0, steps=args.steps, warmup=args.warmup, step_budget=budget)
    value = o["bytes_per_rep"] * o["reps"] / o["seconds"] / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * o["seconds"] / o["reps"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[HEADLINE], "step": "oracle slot write + attention",
                   "parallelism": "single CPU core"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{o['requests']} of 256 requests per step (every "
                                   f"{o['stride']}th), each with its own blocks"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))


def run_ncu_case(spec_arg: str, iters: int = 3, fp8: bool = False) -> None:
    """A small step for profilers: `NAME` or `NAME:N` (the first N requests of
    workload NAME); runs pa_cache_write + pa_forward `iters` times (over an FP8
    cache with scales 0.01 when fp8)."""
    import torch

    import paged_kv_attention_04_gb300 as P
    from paged_kv_attention_04_gb300 import build
    from paged_kv_attention_04_gb300 import workloads as W
    build.build()
    name, _, n = spec_arg.partition(":")
    spec = W.CONFIGS[name]()
    if n:  # N: the first N requests; -N: the last N
        sl = slice(None, int(n)) if int(n) > 0 else slice(int(n), None)
        spec.seq_lens = spec.seq_lens[sl]
        spec.q_lens = spec.q_lens[sl]
        if spec.sharing is not None:
            spec.sharing = spec.sharing[sl]
    st = W.make_step(spec, device="cuda")
    if fp8:
        st.k_cache = (st.k_cache.float() / 0.01).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        st.v_cache = (st.v_cache.float() / 0.01).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        lay = P.layout_of(st.k_cache, spec.num_q_heads, k_scale=0.01, v_scale=0.01)
    else:
        lay = P.layout_of(st.k_cache, spec.num_q_heads)
    ws = P.alloc_workspace(lay, spec.num_seqs, spec.num_tokens, st.max_seq_len)
    out = torch.empty_like(st.q)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(iters):
        P.pa_cache_write(st.k, st.v, st.slot_mapping, st.k_cache, st.v_cache, lay, status)
        P.pa_forward(st.q, st.k_cache, st.v_cache, st.block_tables, st.seq_lens,
                     st.query_start_loc, st.max_query_len, st.max_seq_len, st.scale, out, ws, lay,
                     status)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    print(json.dumps({"ncu_case": spec_arg, "tokens": spec.num_tokens, "ok": True}))


def free_port() -> int:
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def spawn_replicas(n: int, script: str, argv: list[str], env: dict | None = None) -> int:
    """Run `script argv` as n ranks on this node under torch.distributed.run
    (rendezvous on 127.0.0.1, a free port); the ranks' output passes through.
    Returns the launcher's exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={free_port()}", script, *argv]
    return subprocess.run(cmd, env=env).returncode


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-seconds", type=float, default=10.0)
    ap.add_argument("--oracle-stride", type=int, default=1)
    ap.add_argument("--oracle-offset", type=int, default=0, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-sync", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--ncu-case", default=None,
                    help="run a small step for a profiler: NAME, NAME:N (first N requests) "
                         "or NAME:-N (last N)")
    ap.add_argument("--fp8-kv", action="store_true", help="with --ncu-case: an FP8 (E4M3) cache")
    ap.add_argument("--oracle-budget", type=float, default=1.0, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-worker", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.ncu_case:
        run_ncu_case(args.ncu_case, fp8=args.fp8_kv)
        return
    if args.oracle_worker:
        oracle_worker(args.oracle_worker, args.oracle_seconds, args.oracle_stride, args.steps,
                      args.warmup, args.oracle_budget, args.oracle_offset, args.oracle_sync)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference_arm(args)
    elif args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU: start the ranks here (barrier and max-over-ranks
        # timing happen inside each rank's run)
        sys.exit(spawn_replicas(args.gpus, os.path.abspath(__file__), sys.argv[1:]))
    else:
        run_gpu_arm(args)


if __name__ == "__main__":
    main()
