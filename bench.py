"""Benchmark: one decode step of one layer on the LLaMA-13B-shaped batch.

A step is the whole paged decode path for one batch: slot mapping of each
sequence's new token, the cache write of its K/V rows, paged attention decode
(partitioned with the log-sum-exp merge where the lengths call for it) and,
on batches that share prefix blocks, the copy-on-write block copy.  Inputs are
resident in HBM; consecutive timed steps read two KV pools of the batch's shape
(two layers' caches, each larger than L2), so every step is L2-cold (--l2 flush
writes 256 MiB before each step instead).

Prints one JSON line.  value = algorithmic bytes of the step / step time (GB/s);
tokens/s/layer = sequences / step time.  --impl reference times the CPU oracle
(fp64, on the host cores) on a bounded sample of the same batch instead.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload llama13b_b16]
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_293_gb300 import accounting, workloads  # noqa: E402

METRIC = ("paged decode attention HBM GB/s (% of GB300 peak) and decode tokens/s per layer")
FLUSH_BYTES = 256 << 20
LENGTH_RECIPES = {
    "tiny": "fixed {1,17,50,100}",
    "llama7b": "uniform [128, 2048]",
    "llama13b_b16": "lognormal median 512 sigma 1, rounded, clipped [16, 4096]",
    "llama13b_b32": "lognormal median 512 sigma 1, rounded, clipped [16, 4096]",
    "gqa_prefix": "512 shared + uniform [64, 2048] private",
    "long_splitk": "uniform [32768, 131072]",
    "system_prompt": "2048 shared + uniform [16, 256] private",
}
DEFAULT_WORKLOAD = "llama13b_b16"


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def read_traffic(workload):
    """DRAM bytes per launch of the dominant kernel from the committed ncu record of this
    workload, or None when there is none or the kernel source it names has changed since."""
    import hashlib
    summ = os.path.join(ROOT, "profiles", "decode_%s_traffic.txt" % workload)
    if not os.path.exists(summ):
        return None
    vals = {}
    with open(summ) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    h = hashlib.sha256()
    for name in vals.get("source_files", "").split():
        with open(os.path.join(ROOT, "paged_kv_cache_293_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    if vals.get("source_sha256") != h.hexdigest():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class _Nvml:
    """Read-only NVML queries through ctypes: the SM clock and the clock-event (throttle)
    reasons, fast enough to poll every millisecond during a short timed region."""
    SM = 1   # NVML_CLOCK_SM
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown"}

    def __init__(self, uuid, index):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        rc = self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) if uuid else 1
        if rc != 0:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h))
        if rc != 0:
            raise OSError("no NVML handle")
        try:
            self._reasons = self.lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self._reasons = self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.max_mhz = (mx.value if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.SM,
                                                                       ctypes.byref(mx)) == 0
                        else None)

    def close(self):
        self.lib.nvmlShutdown()

    def sample(self):
        c, r = self.ct.c_uint(), self.ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.SM, self.ct.byref(c)) != 0:
            return None
        self._reasons(self.h, self.ct.byref(r))
        return float(c.value), [n for bit, n in self.REASON_BITS.items() if r.value & bit]


class ClockSampler:
    """SM clocks and throttle reasons of this GPU, read (never set) two ways:

    - `nvidia-smi -lms 50` runs from start() to stop() (warm-up, timed region and the
      end-to-end leg: the whole GPU phase), each sample stamped by nvidia-smi itself;
    - inside timed() an NVML poll every millisecond, so that even a timed region of a few
      milliseconds has samples of its own.

    summary() gives the timed region's median clock and the reasons seen in it (NVML
    samples, else the nvidia-smi samples stamped inside it), and the whole phase's median
    over the samples taken under load."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device):
        self.index = device.index or 0
        try:
            u = str(torch.cuda.get_device_properties(device).uuid)
            self.uuid = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            self.uuid = None
        self.proc = None
        self.lines = []          # (wall time from nvidia-smi's stamp, fields)
        self.fast = []           # (wall time, sm MHz, reasons) from NVML inside timed()
        self.windows = []
        try:
            self.nvml = _Nvml(self.uuid, self.index)
        except Exception:
            self.nvml = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.uuid or str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        import datetime
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            try:
                t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except (ValueError, IndexError):
                t = time.time()
            self.lines.append((t, parts[1:]))

    def wait_first(self, timeout=5.0):
        """Block until nvidia-smi has delivered a sample (or the timeout passes)."""
        t = time.time()
        while self.proc is not None and not self.lines and time.time() - t < timeout:
            time.sleep(0.02)

    def timed(self):
        sampler = self

        class _Window:
            def __enter__(self):
                self.stop = threading.Event()
                self.t0 = time.time()
                if sampler.nvml is not None:
                    self.th = threading.Thread(target=self._poll, daemon=True)
                    self.th.start()
                return self

            def _poll(self):
                while not self.stop.is_set():
                    r = sampler.nvml.sample()
                    if r is not None:
                        sampler.fast.append((time.time(), r[0], r[1]))
                    self.stop.wait(0.001)

            def __exit__(self, *exc):
                self.stop.set()
                if sampler.nvml is not None:
                    self.th.join(timeout=2)
                sampler.windows.append((self.t0, time.time()))
        return _Window()

    def stop(self):
        if self.nvml is not None:
            self.nvml.close()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def __enter__(self):
        self.start()
        self._win = self.timed()
        self._win.__enter__()
        return self

    def __exit__(self, *exc):
        self._win.__exit__(*exc)
        self.stop()

    def _smi(self):
        out = []
        for t, parts in self.lines:
            if len(parts) < 8:
                continue
            try:
                sm, mx = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            try:
                util = float(parts[2])
            except ValueError:
                util = 100.0
            rs = [n for n, v in zip(self.NAMES, parts[4:8]) if v.lower().startswith("active")]
            out.append((t, sm, mx, util, rs))
        return out

    def summary(self):
        smi = self._smi()
        if not smi and not self.fast:
            return None
        inside = lambda t: any(a <= t <= b for a, b in self.windows)
        if self.fast:
            timed = [(sm, rs) for t, sm, rs in self.fast]
            source = "NVML every 1 ms inside the timed region"
        else:
            timed = [(sm, rs) for t, sm, mx, u, rs in smi if inside(t)]
            source = "nvidia-smi every 50 ms inside the timed region"
        load = [(sm, rs) for t, sm, mx, u, rs in smi if u >= 50.0] or \
               [(sm, rs) for t, sm, mx, u, rs in smi]
        mx = [m for _, _, m, _, _ in smi] + ([self.nvml.max_mhz] if self.nvml and
                                              self.nvml.max_mhz else [])
        phase = {"sm_mhz": statistics.median(x for x, _ in load) if load else None,
                 "reasons": sorted({r for _, rs in load for r in rs}), "samples": len(load),
                 "source": "nvidia-smi every 50 ms, warm-up to end of the e2e leg, samples with "
                           "GPU utilisation >= 50 %"}
        med = statistics.median(x for x, _ in timed) if timed else phase["sm_mhz"]
        return {"sm_mhz": med, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted({r for _, rs in timed for r in rs} | set(phase["reasons"])),
                "samples": len(timed),
                "source": source if timed else "no sample inside the timed region: whole phase",
                "phase": phase}


def dist_setup(gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class Step:
    """Device buffers and the launch sequence of one decode step through the binding."""

    def __init__(self, P, w, device, fused=True, cascade=False):
        self.P, self.w, self.dev, self.fused = P, w, device, fused
        # batches whose sequences share prefix blocks: the prefix's attention once per kv
        # head on tensor cores, then each sequence's own suffix, then the merge
        self.prefix_len = (len(w.shared_blocks) * w.block_size
                           if cascade and len(w.shared_blocks) and w.dtype != "f32" else 0)
        i32 = lambda a: torch.as_tensor(np.ascontiguousarray(a, np.int32), device=device)
        self.bt = i32(w.block_tables)
        self.pos = i32(w.positions)
        self.ctx = i32(w.context_lens)
        self.pairs = i32(w.cow_pairs) if len(w.cow_pairs) else None
        self.slots = torch.empty(w.num_seqs, dtype=torch.int64, device=device)
        self.out = torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=w.q.dtype,
                               device=device)
        self.mcl = w.max_context_len
        self.psize = w.partition_size or P.pkv_choose_partition_size(
            w.k_pool, w.num_seqs, w.num_q_heads, self.mcl)
        if self.prefix_len:
            self.psize = w.partition_size
            nbytes = P.pkv_cascade_workspace_bytes(w.k_pool, w.num_seqs, w.num_q_heads, self.mcl,
                                                   self.prefix_len, self.psize)
        else:
            nbytes = P.pkv_decode_workspace_bytes(w.k_pool, w.num_seqs, w.num_q_heads, self.mcl,
                                                  self.psize)
        self.ws = P.workspace_tensor(nbytes, device) if nbytes else None
        self.split = nbytes > 0
        if self.prefix_len:
            self.launches = 3 + (0 if fused else 2) + (1 if self.pairs is not None else 0)
        else:
            self.launches = ((1 if fused else 3) + (1 if self.split else 0)
                             + (1 if self.pairs is not None else 0))

    def pre_decode(self):
        """Work before the decode call: the copy-on-write copy, and unless the append is
        fused into the decode launch, slot mapping and the cache write."""
        P, w = self.P, self.w
        if self.pairs is not None:
            P.pkv_copy_blocks(w.k_pool, w.v_pool, self.pairs)
        if not self.fused:
            P.pkv_slot_mapping(self.bt, self.pos, w.block_size, self.slots)
            P.pkv_kv_cache_write(w.k_pool, w.v_pool, w.k_new, w.v_new, self.slots)

    def decode(self):
        """The decode call; fused: it also computes each new token's slot and writes its
        K/V rows (one launch instead of three, same result)."""
        P, w = self.P, self.w
        if self.prefix_len:
            app = dict(k_new=w.k_new, v_new=w.v_new, slot_mapping=self.slots) if self.fused else {}
            P.pkv_paged_attention_decode_cascade(w.q, w.k_pool, w.v_pool, self.bt, self.ctx,
                                                 w.scale, self.out, self.mcl, self.prefix_len,
                                                 self.ws, self.psize, **app)
        elif self.fused:
            P.pkv_paged_attention_decode_append(w.q, w.k_pool, w.v_pool, w.k_new, w.v_new, self.bt,
                                                self.ctx, w.scale, self.out, self.mcl, self.psize,
                                                self.ws, slot_mapping=self.slots)
        else:
            P.pkv_paged_attention_decode(w.q, w.k_pool, w.v_pool, self.bt, self.ctx, w.scale,
                                         self.out, self.mcl, self.psize, self.ws)


def step_bytes(w, psize):
    e = workloads.ELEM_BYTES[w.dtype]
    unique = None
    if len(w.shared_blocks):
        toks = int(w.context_lens.sum()) - (w.num_seqs - 1) * len(w.shared_blocks) * w.block_size
        unique = toks
    dec_logical = accounting.decode_bytes(w.context_lens, w.num_kv_heads, w.num_q_heads,
                                          w.head_dim, e, e, w.block_size, psize)
    dec_unique = accounting.decode_bytes(w.context_lens, w.num_kv_heads, w.num_q_heads,
                                         w.head_dim, e, e, w.block_size, psize,
                                         unique_tokens=unique)
    other = accounting.write_bytes(w.num_seqs, w.num_kv_heads, w.head_dim, e) + 12 * w.num_seqs
    if len(w.cow_pairs):
        other += accounting.copy_bytes(len(w.cow_pairs), w.num_kv_heads, w.block_size,
                                       w.head_dim, e)
    return dec_logical, dec_unique, other


def l2_mode_for(w, args):
    """How the GPU arm keeps its timed steps L2-cold on this batch: two pools alternate, or
    (a pool smaller than twice the L2 would not be evicted by alternating) a flush."""
    return args.l2 if 2 * (w.k_pool.nbytes + w.v_pool.nbytes) > FLUSH_BYTES else "flush"


def workload_config(w, args, world):
    """The `config` of the JSON line: the batch both arms run (the GPU arm and the oracle
    arm print the same dict for the same flags)."""
    return {
        "workload": w.name, "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
        "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
        "context_lens": LENGTH_RECIPES.get(args.workload, ""),
        "mean_context": round(float(w.context_lens.mean()), 1),
        "max_context": w.max_context_len, "pool_blocks": w.num_blocks,
        "kv_bytes_per_step": int(w.context_lens.sum()) * accounting.kv_bytes_per_token(
            w.num_kv_heads, w.head_dim, workloads.ELEM_BYTES[w.dtype]),
        "l2": ("GPU arm: consecutive steps alternate between two KV pools of this shape (two "
               "layers' caches, each larger than L2)" if l2_mode_for(w, args) == "alternate" else
               "GPU arm: flushed by a 256 MiB write before every timed step (outside the "
               "events)"),
        "parallelism": "replicas, one batch per GPU" if world > 1 else "single GPU",
        "seed": args.seed,
        "order": ("the given order" if getattr(args, "order", "given") == "given" else
                  "the shortest fifth of the sequences last, longest of them first"),
    }


def cpu_oracle_rate(w, budget_s=12.0, max_single_s=30.0):
    """Time the oracle (as it stands) on host copies of a bounded sample of the batch."""
    import oracle
    k = workloads.storage_numpy(w.k_pool)
    v = workloads.storage_numpy(w.v_pool)
    q = workloads.storage_numpy(w.q)
    bt, ctx = w.block_tables, w.context_lens
    # calibrate on the first few sequences, then size the sample
    n0 = min(4, w.num_seqs)
    t = time.perf_counter()
    oracle.paged_decode(w.dtype, k, v, q[:n0], bt[:n0], ctx[:n0], w.scale)
    per_tok = (time.perf_counter() - t) / max(1, int(ctx[:n0].sum()))
    n = w.num_seqs
    while n > 1 and per_tok * int(ctx[:n].sum()) > max_single_s:
        n //= 2
    reps, elapsed = 0, 0.0
    t = time.perf_counter()
    while elapsed < budget_s or reps == 0:
        oracle.paged_decode(w.dtype, k, v, q[:n], bt[:n], ctx[:n], w.scale)
        reps += 1
        elapsed = time.perf_counter() - t
        if reps >= 50:
            break
    sec = elapsed / reps
    e = workloads.ELEM_BYTES[w.dtype]
    b = accounting.decode_bytes(ctx[:n], w.num_kv_heads, w.num_q_heads, w.head_dim, e, e,
                                w.block_size)
    return {"gbs": b / sec / 1e9, "tok_s": n / sec, "sec_per_pass": sec, "seqs": n, "reps": reps,
            "cores": oracle.num_threads()}


def run_ours(args):
    world, rank, local = dist_setup(args.gpus)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from paged_kv_cache_293_gb300 import _build
    if rank == 0:
        _build.build()
    barrier(world)
    from paged_kv_cache_293_gb300 import pagedkv as P

    w = workloads.make(args.workload, seed=args.seed + rank, device=device)
    if args.order == "shortest-last":   # the batch order a serving engine can choose
        w = workloads.reorder(w, workloads.shortest_last_order(w.context_lens))
    st = Step(P, w, device, fused=not args.unfused, cascade=args.cascade)
    # Keep every timed step L2-cold: by default consecutive steps read two KV pools of the
    # batch's shape (two layers' caches, each larger than L2); --l2 flush instead writes
    # 256 MiB before each step (outside the events), which leaves dirty lines in L2 that the
    # timed step then has to write back.
    # (a pool smaller than twice the L2 is flushed instead: alternating would not evict it)
    l2_mode = l2_mode_for(w, args)
    pools = [(w.k_pool, w.v_pool), (w.k_pool.clone(), w.v_pool.clone())]
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device) if l2_mode == "flush" else None
    stream = torch.cuda.current_stream(device)

    def prepare(i):
        if flush is not None:
            flush.zero_()
            w.k_pool, w.v_pool = pools[0]
        else:
            w.k_pool, w.v_pool = pools[i % 2]

    clocks = ClockSampler(device).start()
    clocks.wait_first()
    for i in range(args.warmup):
        prepare(i)
        st.pre_decode()
        st.decode()
    torch.cuda.synchronize(device)
    if P.pkv_get_device_error():
        raise RuntimeError("device error flags set during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(device)
    with clocks.timed():
        t_wall = time.perf_counter()
        for i in range(args.steps):
            prepare(i)
            e0, e1, e2 = evs[i]
            e0.record(stream)
            st.pre_decode()
            e1.record(stream)
            st.decode()
            e2.record(stream)
        torch.cuda.synchronize(device)
        wall = time.perf_counter() - t_wall
    barrier(world)
    step_ms = sum(a.elapsed_time(c) for a, _, c in evs) / args.steps
    dec_ms = sum(b.elapsed_time(c) for _, b, c in evs) / args.steps
    step_ms_max = max_over_ranks(step_ms, world, device)
    if P.pkv_get_device_error():
        raise RuntimeError("device error flags set during the timed steps")

    # end to end through the binding with host buffers: H2D inputs, the step, D2H output
    e2e = run_e2e(P, w, st, args, device, pools)
    w.k_pool, w.v_pool = pools[0]
    clocks.stop()
    e2e_ms_max = max_over_ranks(e2e["ms"], world, device)

    dec_logical, dec_unique, other = step_bytes(w, st.psize if st.split and not st.prefix_len else 0)
    if st.prefix_len:  # the cascade's partials: a prefix slot per row plus the suffix partitions
        p_suffix = st.psize or P.pkv_choose_partition_size(w.k_pool, w.num_seqs, w.num_q_heads,
                                                           st.mcl - st.prefix_len)
        extra = accounting.cascade_workspace_bytes(w.context_lens, st.prefix_len, p_suffix,
                                                   w.num_q_heads, w.head_dim)
        dec_logical += extra
        dec_unique += extra
    if st.fused:  # the decode launch also reads the new rows and writes them into the pool
        dec_unique += accounting.write_bytes(w.num_seqs, w.num_kv_heads, w.head_dim,
                                             workloads.ELEM_BYTES[w.dtype])
    total = dec_logical + other
    peak, peak_kind = read_peaks()
    value = world * total / (step_ms_max * 1e-3) / 1e9
    dec_gbs = dec_unique / (dec_ms * 1e-3) / 1e9
    traffic = read_traffic(args.workload)
    tensor = (w.dtype != "f32" and w.num_q_heads // w.num_kv_heads >= 4
              and P.pkv_get_decode_engine() == P.ENGINE_AUTO)
    kernel_name = ("paged_decode_mma_kernel" if tensor else "paged_decode_kernel") + (
        " + lse_merge_kernel" if st.split else "")
    if st.prefix_len:
        kernel_name = "prefix_attention_kernel + " + kernel_name

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        r = cpu_oracle_rate(w)
        cpu = {"value": r["gbs"], "unit": "GB/s", "cores": r["cores"], "kind": "oracle",
               "tokens_per_s_per_layer": r["tok_s"],
               "sample": "first %d of %d sequences of the same batch, %d passes, %.2f s per pass, "
                         "fp64 C with OpenMP" % (r["seqs"], w.num_seqs, r["reps"],
                                                 r["sec_per_pass"])}
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms_max, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "tokens_per_s_per_layer": round(world * w.num_seqs / (step_ms_max * 1e-3), 1),
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        "decode_ms": round(dec_ms, 5),
        "config": workload_config(w, args, world),
        "partition_size": st.psize if st.split else 0,
        "path": ("decode with the append fused (slot, write, attention in one launch)"
                 if st.fused else "slot mapping, cache write, decode: three launches")
                + ("; cascade over the %d-token shared prefix" % st.prefix_len
                   if st.prefix_len else ""),
        "roofline": {
            "kernel": kernel_name,
            "bound": "hbm", "achieved": round(dec_gbs, 2), "peak": peak, "unit": "GB/s",
            "frac": round(dec_gbs / peak, 4), "peak_kind": peak_kind,
            "traffic": traffic, "algorithmic_bytes": dec_unique,
        },
        "cpu_baseline": cpu,
        "e2e": {"value": round(world * total / (e2e_ms_max * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms_max, 5),
                "overlap": "input and output copies on their own stream, two steps deep",
                "l2": "consecutive steps alternate between two KV pools (two layers)",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"]},
        "gpu_launches": st.launches * args.steps,
        "clocks": clocks.summary(),
        "wall_s_timed": round(wall, 3),
    }
    print(json.dumps(line), flush=True)


def _e2e_two_deep(device, dev_src, out_like, step, warmup, steps):
    """End-to-end timing through the binding: every step copies its inputs (`dev_src`, a
    dict of device tensors whose pinned host copy is made here) in from pinned host memory,
    in one copy, and reads its output back.  As a serving loop would, the copies run on their own
    stream two steps deep: step i+1's inputs go in while step i computes, and step i's output
    comes back while step i+1 computes.  `step(inputs, out, slot)` launches one step on the
    current stream, reading `inputs` (a dict like `dev_src`) and writing `out`; `slot` (0 or
    1) alternates between steps.  Timed with CUDA events from the first input copy to the
    last output copy; returns ms per step and the bytes copied each way per step."""
    # the inputs packed into one pinned buffer (each at a 256-byte offset), so a step's
    # inputs go in by one copy, as a serving loop that stages them would send them
    offs, total = {}, 0
    for k, v in dev_src.items():
        offs[k] = total
        total += (v.numel() * v.element_size() + 255) // 256 * 256
    host_in = torch.zeros(total, dtype=torch.uint8).pin_memory()
    for k, v in dev_src.items():
        n = v.numel() * v.element_size()
        host_in[offs[k]:offs[k] + n].copy_(v.detach().contiguous().view(-1).view(torch.uint8).cpu())
    dev_in = [torch.empty(total, dtype=torch.uint8, device=device) for _ in range(2)]

    def views(buf):
        return {k: buf[offs[k]:offs[k] + v.numel() * v.element_size()].view(v.dtype).view(v.shape)
                for k, v in dev_src.items()}

    bufs = [views(d) for d in dev_in]
    outs = [torch.empty_like(out_like) for _ in range(2)]
    h_out = [torch.empty(out_like.shape, dtype=out_like.dtype).pin_memory() for _ in range(2)]
    h2d = total
    d2h = h_out[0].numel() * h_out[0].element_size()
    comp = torch.cuda.current_stream(device)
    copy = torch.cuda.Stream(device)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    out_read = [torch.cuda.Event() for _ in range(2)]

    def load(i):
        b = i % 2
        if i >= 2:
            copy.wait_event(computed[b])        # step i - 2 is done with this buffer
        with torch.cuda.stream(copy):
            dev_in[b].copy_(host_in, non_blocking=True)
        in_ready[b].record(copy)

    def run(n):
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        t0.record(copy)
        load(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                load(i + 1)
            comp.wait_event(in_ready[b])
            if i >= 2:
                comp.wait_event(out_read[b])    # step i - 2's output has been read back
            step(bufs[b], outs[b], b)
            computed[b].record(comp)
            copy.wait_event(computed[b])
            with torch.cuda.stream(copy):
                h_out[b].copy_(outs[b], non_blocking=True)
            out_read[b].record(copy)
        t1.record(copy)
        t1.synchronize()
        return t0.elapsed_time(t1) / n

    run(max(3, warmup))
    return {"ms": run(max(3, steps)), "h2d": h2d, "d2h": d2h}


def run_e2e(P, w, st, args, device, pools):
    """The decode step end to end: q, the new K/V rows, block tables, positions and lengths
    in from pinned host memory every step, the output back, two steps deep; consecutive
    steps read two different KV pools of the batch's shape (two layers' caches, each larger
    than L2), so no step finds the previous step's pages in L2."""
    dev_src = {"q": w.q, "k_new": w.k_new, "v_new": w.v_new, "bt": st.bt, "pos": st.pos,
               "ctx": st.ctx}
    saved = (w.q, w.k_new, w.v_new, st.bt, st.pos, st.ctx, st.out, w.k_pool, w.v_pool)

    def step(x, out, b):
        w.q, w.k_new, w.v_new = x["q"], x["k_new"], x["v_new"]
        st.bt, st.pos, st.ctx, st.out = x["bt"], x["pos"], x["ctx"], out
        w.k_pool, w.v_pool = pools[b]
        st.pre_decode()
        st.decode()

    try:
        return _e2e_two_deep(device, dev_src, st.out, step, args.warmup, args.steps // 4)
    finally:
        w.q, w.k_new, w.v_new, st.bt, st.pos, st.ctx, st.out, w.k_pool, w.v_pool = saved


def run_reference(args):
    """The CPU oracle arm: rank 0 only, bounded samples of the same batch on host cores."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    w = workloads.make(args.workload, seed=args.seed, device="cpu")
    k = workloads.storage_numpy(w.k_pool)
    v = workloads.storage_numpy(w.v_pool)
    q = workloads.storage_numpy(w.q)
    kn, vn = workloads.storage_numpy(w.k_new), workloads.storage_numpy(w.v_new)
    bt, ctx, pos = w.block_tables, w.context_lens, w.positions
    # size each step so that warm-up + timed steps take a few minutes at most
    per_step_budget = max(0.05, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    t = time.perf_counter()
    oracle.paged_decode(w.dtype, k, v, q[:2], bt[:2], ctx[:2], w.scale)
    per_tok = (time.perf_counter() - t) / max(1, int(ctx[:2].sum()))
    n = 1
    while n < w.num_seqs and per_tok * int(ctx[:n + 1].sum()) <= per_step_budget:
        n += 1

    def one_step():
        slots = oracle.slot_mapping(bt[:n], pos[:n], w.block_size)
        oracle.kv_cache_write(w.dtype, k, v, kn[:n], vn[:n], slots)
        oracle.paged_decode(w.dtype, k, v, q[:n], bt[:n], ctx[:n], w.scale)

    for _ in range(args.warmup):
        one_step()
    t = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    sec = (time.perf_counter() - t) / args.steps
    e = workloads.ELEM_BYTES[w.dtype]
    b = accounting.decode_bytes(ctx[:n], w.num_kv_heads, w.num_q_heads, w.head_dim, e, e,
                                w.block_size) + accounting.write_bytes(n, w.num_kv_heads,
                                                                       w.head_dim, e)
    value = b / sec / 1e9
    sample = ("first %d of %d sequences of the %s batch per step (slot mapping, cache write, "
              "decode), fp64 C with OpenMP" % (n, w.num_seqs, w.name))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "tokens_per_s_per_layer": round(n / sec, 2),
        "config": workload_config(w, args, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "kind": "oracle",
                         "cores": oracle.num_threads(), "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ the other rows of the path

def _time_steps(device, stream, steps, warmup, prepare, body):
    """warm-up, then `steps` timed calls of body() with CUDA events on `stream`; mean ms."""
    for i in range(warmup):
        prepare(i)
        body()
    torch.cuda.synchronize(device)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    with ClockSampler(device) as clocks:
        for i in range(steps):
            prepare(i)
            evs[i][0].record(stream)
            body()
            evs[i][1].record(stream)
        torch.cuda.synchronize(device)
    if not steps:
        return 0.0, None
    return sum(a.elapsed_time(b) for a, b in evs) / steps, clocks.summary()


def _base_line(args, metric, value, unit, ms, dtype, config, roofline, cpu, e2e, launches, clocks,
               higher=True):
    return {"metric": metric, "value": round(value, 3), "unit": unit, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": higher, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
            "data": "synthetic", "config": config, "roofline": roofline, "cpu_baseline": cpu,
            "e2e": e2e, "gpu_launches": launches, "clocks": clocks}


def run_multi(args):
    """Several new tokens per sequence (a speculative draft being verified, or a chunked
    prefill's tail): their K/V rows written into the cache and the causal multi-query paged
    decode, in one launch (with --unfused: slot mapping, cache write, then the decode).
    value = algorithmic bytes / step time."""
    import oracle
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    from paged_kv_cache_293_gb300 import _build
    _build.build()
    from paged_kv_cache_293_gb300 import pagedkv as P
    w = workloads.make(args.workload, seed=args.seed, device=device)
    nq, S = args.queries, w.num_seqs
    if int(w.context_lens.min()) < nq:
        raise SystemExit("every context must hold the %d new tokens" % nq)
    g = torch.Generator(device=device).manual_seed(args.seed + 7)
    tdt = w.q.dtype
    q = torch.randn((S, nq, w.num_q_heads, w.head_dim), generator=g, device=device).to(tdt)
    k_new = torch.randn((S * nq, w.num_kv_heads, w.head_dim), generator=g, device=device).to(tdt)
    v_new = torch.randn((S * nq, w.num_kv_heads, w.head_dim), generator=g, device=device).to(tdt)
    i32 = lambda a: torch.as_tensor(np.ascontiguousarray(a, np.int32), device=device)
    pos_np = (w.context_lens[:, None] - nq + np.arange(nq)[None, :]).reshape(-1)
    pos, tseq = i32(pos_np), i32(np.repeat(np.arange(S), nq))
    bt, ctx = i32(w.block_tables), i32(w.context_lens)
    slots = torch.empty(S * nq, dtype=torch.int64, device=device)
    out = torch.empty_like(q)
    mcl = w.max_context_len
    ws_bytes = P.pkv_decode_workspace_bytes(w.k_pool, S * nq, w.num_q_heads, mcl, 0)
    ws = P.workspace_tensor(ws_bytes, device) if ws_bytes else None
    pools = [(w.k_pool, w.v_pool), (w.k_pool.clone(), w.v_pool.clone())]
    cur = {}

    def prepare(i):
        cur["k"], cur["v"] = pools[i % 2]

    dev_in = {"q": q, "k_new": k_new, "v_new": v_new, "bt": bt, "ctx": ctx}
    if args.unfused:   # the fused launch derives the positions from the lengths
        dev_in.update(pos=pos, tseq=tseq)

    def launch(x, o, kp, vp):
        if args.unfused:
            P.pkv_slot_mapping(x["bt"], x["pos"], w.block_size, slots, token_seq=x["tseq"])
            P.pkv_kv_cache_write(kp, vp, x["k_new"], x["v_new"], slots)
            P.pkv_paged_attention_decode_multi(x["q"], kp, vp, x["bt"], x["ctx"], w.scale, o, mcl,
                                               0, ws)
        else:
            P.pkv_paged_attention_decode_multi_append(x["q"], kp, vp, x["k_new"], x["v_new"],
                                                      x["bt"], x["ctx"], w.scale, o, mcl, 0, ws,
                                                      slot_mapping=slots)

    def body():
        launch(dev_in, out, cur["k"], cur["v"])

    stream = torch.cuda.current_stream(device)
    ms, clocks = _time_steps(device, stream, args.steps, args.warmup, prepare, body)
    if P.pkv_get_device_error():
        raise RuntimeError("device error flags set")
    e = workloads.ELEM_BYTES[w.dtype]
    kv = int(w.context_lens.sum()) * accounting.kv_bytes_per_token(w.num_kv_heads, w.head_dim, e)
    qo = 2 * S * nq * w.num_q_heads * w.head_dim * e
    table = int(np.ceil(w.context_lens / w.block_size).sum()) * 4
    write = accounting.write_bytes(S * nq, w.num_kv_heads, w.head_dim, e) + 12 * S * nq
    total = kv + qo + table + write    # partition partials not counted
    peak, peak_kind = read_peaks()

    # the same step end to end: q, the new rows, tables, lengths and positions in from
    # pinned host memory every step, out back, two steps deep
    e2e = _e2e_two_deep(device, dev_in, out,
                        lambda x, o, b: launch(x, o, pools[b][0], pools[b][1]),
                        args.warmup, args.steps // 4)
    e2e_ms, h2d, d2h = e2e["ms"], e2e["h2d"], e2e["d2h"]

    cpu = None
    if not args.no_cpu_baseline:
        k_h, v_h = workloads.storage_numpy(pools[0][0]), workloads.storage_numpy(pools[0][1])
        q_h = workloads.storage_numpy(q)
        n = S
        t = time.perf_counter()
        oracle.paged_decode_multi(w.dtype, k_h, v_h, q_h[:2], w.block_tables[:2],
                                  w.context_lens[:2], w.scale)
        per_tok = (time.perf_counter() - t) / max(1, int(w.context_lens[:2].sum()))
        while n > 1 and per_tok * int(w.context_lens[:n].sum()) > 15.0:
            n //= 2
        t = time.perf_counter()
        oracle.paged_decode_multi(w.dtype, k_h, v_h, q_h[:n], w.block_tables[:n],
                                  w.context_lens[:n], w.scale)
        sec = time.perf_counter() - t
        b = int(w.context_lens[:n].sum()) * accounting.kv_bytes_per_token(
            w.num_kv_heads, w.head_dim, e)
        cpu = {"value": round(b / sec / 1e9, 4), "unit": "GB/s", "cores": oracle.num_threads(),
               "kind": "oracle", "tokens_per_s_per_layer": round(n * nq / sec, 2),
               "sample": "first %d of %d sequences, %d queries each, one pass of %.2f s, fp64 C "
                         "with OpenMP" % (n, S, nq, sec)}
    dec_name = "paged_decode_mma_kernel" if (w.dtype != "f32") else "paged_decode_kernel"
    line = _base_line(
        args, "multi-query paged decode HBM GB/s and new tokens/s per layer",
        total / (ms * 1e-3) / 1e9, "GB/s", ms, w.dtype,
        {"workload": w.name + "_q%d" % nq, "num_seqs": S, "queries_per_seq": nq,
         "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
         "block_size": w.block_size, "context_lens": LENGTH_RECIPES.get(args.workload, ""),
         "kv_bytes_per_step": kv, "partition_size": "auto",
         "l2": "consecutive steps alternate between two KV pools (two layers' caches)",
         "path": ("slot mapping and cache write of the %d new tokens per sequence, causal "
                  "multi-query decode" % nq) if args.unfused else
                 ("the %d new tokens per sequence written into the cache by the causal "
                  "multi-query decode launch itself" % nq)},
        {"kernel": dec_name + " (all launches of the step)", "bound": "hbm",
         "achieved": round(total / (ms * 1e-3) / 1e9, 2), "peak": peak, "unit": "GB/s",
         "frac": round(total / (ms * 1e-3) / 1e9 / peak, 4), "peak_kind": peak_kind,
         # DRAM bytes per decode launch (the step's dominant kernel) from the committed
         # ncu record of the fused step, when there is one for this source
         "traffic": None if args.unfused else read_traffic("multi%d_%s" % (nq, args.workload)),
         "algorithmic_bytes": total},
        cpu,
        {"value": round(total / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
         "ms_per_step": round(e2e_ms, 5),
         "overlap": "input and output copies on their own stream, two steps deep",
         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        ((3 if args.unfused else 1) + (1 if ws_bytes else 0)) * args.steps, clocks)
    line["tokens_per_s_per_layer"] = round(S * nq / (ms * 1e-3), 1)
    print(json.dumps(line), flush=True)


def run_swap(args):
    """Preemption swap: a quarter of the batch's blocks out to a pinned host pool and back.
    The denominator is the same bytes moved by cudaMemcpyAsync between contiguous pinned
    host memory and the device, measured in the same run."""
    import oracle
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    from paged_kv_cache_293_gb300 import _build
    _build.build()
    from paged_kv_cache_293_gb300 import pagedkv as P
    w = workloads.make(args.workload, seed=args.seed, device=device)
    used = np.unique(np.concatenate([w.block_tables[s, :-(-int(c) // w.block_size)]
                                     for s, c in enumerate(w.context_lens)]))
    rng = np.random.default_rng(args.seed + 11)
    moved = np.sort(rng.choice(used, size=max(1, len(used) // 4), replace=False)).astype(np.int32)
    n = len(moved)
    shape = (n,) + tuple(w.k_pool.shape[1:])
    hk = torch.empty(shape, dtype=w.k_pool.dtype).pin_memory()
    hv = torch.empty(shape, dtype=w.v_pool.dtype).pin_memory()
    out_pairs = torch.as_tensor(np.stack([moved, np.arange(n, dtype=np.int32)], 1).reshape(-1),
                                device=device)
    in_pairs = torch.as_tensor(np.stack([np.arange(n, dtype=np.int32), moved], 1).reshape(-1),
                               device=device)
    nbytes = 2 * hk.numel() * hk.element_size()          # both pools, one direction
    stream = torch.cuda.current_stream(device)
    idx = torch.as_tensor(moved, device=device).long()
    before = (w.k_pool[idx].cpu(), w.v_pool[idx].cpu())

    def body():
        P.pkv_swap_blocks(w.k_pool, w.v_pool, hk, hv, out_pairs)
        P.pkv_swap_blocks(hk, hv, w.k_pool, w.v_pool, in_pairs)

    ms, clocks = _time_steps(device, stream, args.steps, args.warmup, lambda i: None, body)
    if P.pkv_get_device_error():
        raise RuntimeError("device error flags set")
    same = (torch.equal(w.k_pool[idx].cpu(), before[0])
            and torch.equal(w.v_pool[idx].cpu(), before[1]))
    # the link's own rate for the same bytes: contiguous pinned copies each way
    dk = torch.empty(shape, dtype=w.k_pool.dtype, device=device)
    dv = torch.empty_like(dk)

    def copies():
        hk.copy_(dk, non_blocking=True)
        hv.copy_(dv, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)

    link_ms, _ = _time_steps(device, stream, args.steps, args.warmup, lambda i: None, copies)
    value = 2 * nbytes / (ms * 1e-3) / 1e9
    link = 2 * nbytes / (link_ms * 1e-3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        k_h, v_h = workloads.storage_numpy(w.k_pool), workloads.storage_numpy(w.v_pool)
        hk2 = np.empty((n,) + k_h.shape[1:], k_h.dtype)
        hv2 = np.empty_like(hk2)
        pairs = np.stack([moved, np.arange(n, dtype=np.int32)], 1)
        t = time.perf_counter()
        reps = 0
        while time.perf_counter() - t < 5.0 or reps == 0:
            oracle.swap_blocks(k_h, v_h, hk2, hv2, pairs)
            reps += 1
        sec = (time.perf_counter() - t) / reps
        cpu = {"value": round(nbytes / sec / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": "the same %d blocks copied out on the host (one direction), %d passes"
                         % (n, reps)}
    line = _base_line(
        args, "block swap GPU <-> pinned host GB/s (both directions)", value, "GB/s", ms,
        w.dtype,
        {"workload": w.name + "_swap", "blocks_moved": n, "pool_blocks": w.num_blocks,
         "bytes_each_way": nbytes, "block_choice": "a seeded quarter of the blocks in use",
         "round_trip_bit_exact": bool(same), "path": "swap out, then swap back in"},
        {"kernel": "copy_blocks_kernel (two launches)", "bound": "host link",
         "achieved": round(value, 2), "peak": round(link, 2), "unit": "GB/s",
         "frac": round(value / link, 4),
         "peak_kind": "measured in this run: cudaMemcpyAsync of the same bytes, contiguous "
                      "pinned host <-> device, both directions", "traffic": None,
         "algorithmic_bytes": 2 * nbytes},
        cpu,
        {"value": round(value, 2), "unit": "GB/s", "ms_per_step": round(ms, 5),
         "note": "the swap moves host buffers by itself: this is the call a user makes",
         "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes},
        2 * args.steps, clocks)
    print(json.dumps(line), flush=True)


def run_alloc(args):
    """Block bookkeeping of one decode step on the device: every sequence grows by one token
    (a new block where it crosses a block boundary).  Latency-bound; the floor is the
    library's smallest launch (slot mapping of one token) timed in the same run."""
    import oracle
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    from paged_kv_cache_293_gb300 import _build
    _build.build()
    from paged_kv_cache_293_gb300 import pagedkv as P
    w = workloads.make(args.workload, seed=args.seed, device=device)
    S, B = w.num_seqs, w.block_size
    steps_total = args.warmup + args.steps
    M = int(-(-(int(w.context_lens.max()) + steps_total) // B)) + 1
    need = int(np.sum(-(-(w.context_lens + steps_total) // B))) + 16
    N = max(need, 1024)
    # a small pool: no block is shared, so no copy-on-write copies are made
    kp = torch.empty((N, w.num_kv_heads, B, w.head_dim), dtype=w.k_pool.dtype, device=device)
    vp = torch.empty_like(kp)
    alloc = P.BlockAllocator(N, device)
    P.pkv_allocator_reset(alloc)
    tables = torch.full((S, M), -1, dtype=torch.int32, device=device)
    status = torch.empty(S, dtype=torch.int32, device=device)
    i32 = lambda a: torch.as_tensor(np.ascontiguousarray(a, np.int32), device=device)
    lens = [i32(w.context_lens + i) for i in range(steps_total + 1)]
    P.pkv_allocate_for_append(alloc, kp, vp, tables, i32(np.zeros(S)), lens[0], status)
    cur = {}

    def prepare(i):
        cur["i"] = i

    def body():
        i = cur["i"]
        P.pkv_allocate_for_append(alloc, kp, vp, tables, lens[i], lens[i + 1], status)

    stream = torch.cuda.current_stream(device)
    # warm-up steps 0..W-1, timed steps W..W+K-1
    ms_w, _ = _time_steps(device, stream, 0, args.warmup, prepare, body)
    base = args.warmup
    ms, clocks = _time_steps(device, stream, args.steps, 0, lambda i: prepare(base + i), body)
    torch.cuda.synchronize(device)
    ok = bool(torch.all(status == 0)) and not P.pkv_get_device_error()
    one_tok = torch.zeros(1, dtype=torch.int32, device=device)
    slot1 = torch.empty(1, dtype=torch.int64, device=device)
    floor_ms, _ = _time_steps(device, stream, args.steps, args.warmup, lambda i: None,
                              lambda: P.pkv_slot_mapping(tables[:1], one_tok, B, slot1))
    new_blocks = int(np.sum(-(-(w.context_lens + steps_total) // B)
                            - -(-(w.context_lens + base) // B)))
    cpu = None
    if not args.no_cpu_baseline:
        ref = oracle.Allocator(N)
        k_h = np.zeros((N, 1), np.uint16)   # no block is shared: nothing is copied
        tb = np.full((S, M), -1, np.int32)
        ref.allocate_for_append(k_h, k_h, B, tb, np.zeros(S, np.int32),
                                w.context_lens.astype(np.int32))
        reps, t = 0, time.perf_counter()
        while reps < steps_total and (time.perf_counter() - t < 5.0 or reps == 0):
            ref.allocate_for_append(k_h, k_h, B, tb, (w.context_lens + reps).astype(np.int32),
                                    (w.context_lens + reps + 1).astype(np.int32))
            reps += 1
        sec = (time.perf_counter() - t) / reps
        cpu = {"value": round(sec * 1e6, 2), "unit": "us per step", "cores": 1, "kind": "oracle",
               "sample": "the same %d sequences growing one token a step, %d steps (sequential "
                         "C)" % (S, reps)}
    line = _base_line(
        args, "device block bookkeeping: microseconds per decode step's allocate-for-append",
        ms * 1e3, "us", ms, "int32",
        {"workload": w.name + "_alloc", "num_seqs": S, "block_size": B, "pool_blocks": N,
         "blocks_taken_in_timed_steps": new_blocks,
         "all_statuses_ok": ok,
         "path": "every sequence grows by one token per step; a fresh block where it crosses a "
                 "block boundary"},
        {"kernel": "allocate_for_append_kernel", "bound": "latency", "achieved": round(ms * 1e3, 3),
         "peak": round(floor_ms * 1e3, 3), "unit": "us", "frac": round(floor_ms / ms, 4),
         "peak_kind": "measured in this run: one-token slot mapping launch (the library's "
                      "smallest kernel)", "traffic": None, "algorithmic_bytes": None},
        cpu,
        None, args.steps, clocks, higher=False)
    line["sequences_per_s"] = round(S / (ms * 1e-3), 1)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.CONFIGS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--l2", choices=["alternate", "flush"], default="alternate",
                    help="how timed steps are kept L2-cold")
    ap.add_argument("--cascade", action="store_true",
                    help="shared-prefix batches: prefix attention once per kv head, then the "
                         "suffixes, then the merge (pays when the shared prefix is long against "
                         "the suffixes, as on the system-prompt batch)")
    ap.add_argument("--path", choices=["decode", "multi", "swap", "alloc"], default="decode",
                    help="decode: the decode step (default); multi: several new tokens per "
                         "sequence; swap: blocks to pinned host memory and back; alloc: the "
                         "device block bookkeeping of a step")
    ap.add_argument("--queries", type=int, default=4, help="new tokens per sequence (--path multi)")
    ap.add_argument("--unfused", action="store_true",
                    help="slot mapping, cache write and decode as three launches")
    ap.add_argument("--order", choices=["given", "shortest-last"], default="given",
                    help="sequence order of the batch: as generated (default), or the shortest "
                         "fifth last, the order a serving engine that knows the lengths can pick")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.path == "multi":
        run_multi(args)
    elif args.path == "swap":
        run_swap(args)
    elif args.path == "alloc":
        run_alloc(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
