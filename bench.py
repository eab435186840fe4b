#!/usr/bin/env python3
"""Benchmark of the MatMulNBits hot path on GB300.

Default workload: the int4 decode GEMV, M=1, K=4096, N=11008, bf16 X/Y, f16
scales, uint8 zero points (block 32), metric GB/s (algorithmic bytes / time).
``--config 4`` selects the M=512 prefill GEMM (metric TFLOP/s).  The default
run also reports the M=512 GEMM and the int8-activation path (accuracy level
4: activation quantisation + integer GEMV) on the decode workload and the
grouped mixture-of-experts decode GEMV (``moe``) as secondary objects.

A step is one mnb_matmul call over one batch (the decode step of one
projection).  Weights are rotated over enough distinct copies that every
step streams them from HBM (copies x bytes >= 3 x L2).  The timed steps are
captured into CUDA graphs (all of them in one graph up to 2048 steps; graphs
of 1024 beyond), one kernel node per call as a serving loop would launch
them.  A GPU spin kernel is queued just before the start event, so the host
has submitted every graph before the device reaches the timed region, which
then holds device time only, at any step count.  Timing uses CUDA events on
the launching stream with a barrier and a device synchronise on both sides.
Clocks and throttle reasons are sampled read-only through NVML in-process
around the timed region.  Under torchrun each rank runs its own replica
(weak scaling, no data-path collective); the time is the max over ranks.

The default run also reports, as secondary objects with their own roofline,
the 8-bit K=11008 decode (``int8_k11008``) and the 2-bit M=8 batch
(``int2_m8``).

The ``e2e`` object times the same steps through mnb_matmul_host_io: X starts
in pinned host memory and Y ends there, moved by the library's kernels
inside the timed region.

Prints ONE JSON line on rank 0.  ``--impl reference`` times the CPU oracle
(the reference arm) on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_quantized_weight_matmulnbits_gb300 import workloads as wl  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=20000)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=1)
    ap.add_argument("--kernel", default="auto")
    ap.add_argument("--no-pdl", action="store_true", help="launch without programmatic dependent launch")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--only", default=None, choices=["moe", "fp8", "nvfp4", "act_order", "act_order_m512"],
                    help="diagnostic: time only this secondary object (for profiling its kernel alone)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--accuracy-level", type=int, default=0, choices=[0, 4],
                    help="4: int8-activation path for the main workload")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def metric_of(w: wl.Workload):
    if w.M >= 64:
        return "TFLOP/s", w.flops() / 1e12
    return "GB/s", w.algorithmic_bytes() / 1e9


# ---- clocks ----------------------------------------------------------------

class ClockSampler:
    """Read-only NVML sampling of the SM clock and the clock-event (throttle)
    reasons in a background thread, through the driver's libnvidia-ml (ctypes,
    no Python NVML package needed).  Nothing is ever set."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, period_s: float = 0.0005):
        import ctypes
        import threading
        self.period = period_s
        self.samples = []
        self.err = None
        self._stop = threading.Event()
        self._thread = None
        self.lib = None
        self.handle = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            handle = ctypes.c_void_p()
            uuid = None
            try:
                import torch
                u = str(torch.cuda.get_device_properties(device_index).uuid)
                uuid = u if u.startswith("GPU-") else "GPU-" + u
            except Exception:
                uuid = None
            if uuid is None or lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(handle)) != 0:
                if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device_index), ctypes.byref(handle)) != 0:
                    raise OSError("no NVML handle")
            self.lib, self.handle = lib, handle
            self._reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            mx = ctypes.c_uint()
            self.sm_max = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0 \
                else None
        except (OSError, AttributeError) as e:
            self.err = str(e) or type(e).__name__

    def _read(self):
        import ctypes
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) != 0:
            return None
        if self._reasons_fn(self.handle, ctypes.byref(rs)) != 0:
            rs.value = 0
        return (time.perf_counter(), float(clk.value), int(rs.value))

    def _loop(self):
        while not self._stop.is_set():
            s = self._read()
            if s is not None:
                self.samples.append(s)
            time.sleep(self.period)

    def start(self):
        import threading
        if self.lib is None:
            return
        s = self._read()
        if s is not None:
            self.samples.append(s)
        self._thread = threading.Thread(target=self._loop, daemon=True)
        self._thread.start()

    def stop(self):
        if self.lib is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [f"NVML unavailable: {self.err}"],
                    "samples": 0, "source": "nvml"}
        self._stop.set()
        if self._thread is not None:
            self._thread.join()
        s = self._read()
        if s is not None:
            self.samples.append(s)
        sm = [c for _, c, _ in self.samples]
        reasons = set()
        for _, _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.sm_max,
                "reasons": sorted(reasons), "samples": len(sm),
                "sm_mhz_min": min(sm) if sm else None,
                "source": "nvml, in-process, from before the pre-spin to after the timed region"}


# ---- CPU oracle timing -----------------------------------------------------

def cpu_oracle_rate(w: wl.Workload, data, seconds: float):
    """Time the oracle (as it stands) on this host's cores over a bounded sample
    of the workload; return (value in the metric's unit, cores, sample text)."""
    import numpy as np
    import oracle
    oracle.build()
    x64 = wl.widen_f64(data["x"], w.act_dtype)
    s32 = wl.widen_f32(data["scales"], w.scale_dtype)
    cores = oracle.threads()
    unit, per_full = metric_of(w)
    # sample: all rows of x against a prefix of the output columns, sized to ~seconds
    n_cols = max(1, min(w.N, 64))
    done_cols, t_total = 0, 0.0
    rng = np.random.default_rng(1)
    while t_total < seconds and done_cols < 1000 * w.N:
        cols = rng.integers(0, w.N, n_cols)
        ms = np.repeat(np.arange(w.M), n_cols)
        ns = np.tile(cols, w.M)
        t0 = time.perf_counter()
        oracle.matmul_points(x64, data["b"], s32, data["zp"], w.N, w.K, w.bits, w.bs, ms, ns)
        dt = time.perf_counter() - t0
        t_total += dt
        done_cols += n_cols
        if dt < 0.5 * seconds / 4:
            n_cols = min(w.N * 8, n_cols * 2)
    frac = done_cols / w.N
    value = per_full * frac / t_total
    sample = (f"{done_cols} output columns x all {w.M} rows (={frac:.3g} of the workload) in {t_total:.2f} s, "
              f"fp64 oracle, OpenMP over outputs")
    return value, cores, sample


# ---- rank logic (replicas: no data-path collective) ------------------------

def max_over_ranks(t: float, dist=None, device="cuda") -> float:
    """The slowest rank's time (the job ends when the last replica does)."""
    if dist is None:
        return t
    import torch
    tt = torch.tensor([t], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def whole_job_value(world: int, steps: int, per_step: float, t: float) -> float:
    """Units all ranks processed / the max-over-ranks time (weak scaling)."""
    return world * steps * per_step / t


# ---- GPU arm ---------------------------------------------------------------

def traffic_for(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source
    it was taken from is unchanged."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e:
        return None
    src = os.path.join(ROOT, e["source"])
    if not os.path.exists(src):
        return None
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return e["bytes_per_launch"] if h == e["source_sha256_16"] else None


def run_ours(args):
    import numpy as np
    import torch

    import block_quantized_weight_matmulnbits_gb300 as mnb

    TORCH_DT = {wl.F32: torch.float32, wl.F16: torch.float16, wl.BF16: torch.bfloat16}

    def to_dev(stored, dtype):
        a = np.ascontiguousarray(stored)
        if dtype == wl.F32:
            return torch.from_numpy(a.astype(np.float32)).cuda()
        return torch.from_numpy(a.view(np.int16)).cuda().view(TORCH_DT[dtype])

    def aligned_empty(nbytes, align=256):
        raw = torch.empty(nbytes + align, dtype=torch.uint8, device="cuda")
        off = (-raw.data_ptr()) % align
        return raw[off:off + nbytes]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    mnb.load()
    pk, pk_src = peaks()

    flags = 0 if args.no_pdl else mnb.MNB_FLAG_PDL

    def replay_timed(call, steps, warmup, stream, per_graph=None):
        """Run `warmup` untimed steps, then time exactly `steps` steps with CUDA
        events on `stream`, barrier + synchronise on both sides.  Steps are
        captured into CUDA graphs of G calls (G = steps when steps <= 2048) so
        that the host launches a handful of graphs at most; a GPU spin kernel
        queued just before the start event holds the device while the host
        submits them, so the timed region holds device work only.  Returns
        (seconds, clocks)."""
        G = per_graph or (steps if steps <= 2048 else 1024)
        with torch.cuda.stream(stream):
            for i in range(min(G, 64)):
                call(i)
        torch.cuda.synchronize()

        def capture(n, first=0):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                for i in range(n):
                    call(first + i)
            return gr

        g = capture(G)
        reps, rem = divmod(steps, G)
        g_rem = capture(rem, reps * G) if rem else None
        wreps, wrem = divmod(warmup, G)
        with torch.cuda.stream(stream):
            for _ in range(wreps):
                g.replay()
            if wrem:
                capture(wrem).replay()
        barrier()
        clocks = ClockSampler(local)
        clocks.start()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        spin_ms = 3.0 + 0.05 * (reps + 1)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(int(spin_ms * 2.2e6))
            ev0.record(stream)
            for _ in range(reps):
                g.replay()
            if g_rem is not None:
                g_rem.replay()
            ev1.record(stream)
        barrier()
        ck = clocks.stop()
        return max_over_ranks(ev0.elapsed_time(ev1) / 1e3, dist), ck

    def measure(w: wl.Workload, steps: int, warmup: int, kernel: str, want_e2e: bool, acc: int = 0,
                act_order: bool = False):
        data = wl.generate(w)
        x = to_dev(data["x"], w.act_dtype)
        b = torch.from_numpy(np.ascontiguousarray(data["b"])).cuda()
        s0 = to_dev(data["scales"], w.scale_dtype)
        zp0 = None if data["zp"] is None else torch.from_numpy(np.ascontiguousarray(data["zp"])).cuda()
        call_flags = flags
        if act_order:
            # act-order weights: a seeded g_idx (a permutation of the depths cut into blocks), packed with
            # the permutation stored in the buffer, run with MNB_FLAG_KPERM
            order = np.random.default_rng(w.seed + 7).permutation(w.K)
            g = np.empty(w.K, dtype=np.int32)
            g[order] = np.arange(w.K, dtype=np.int32) // w.bs
            packed = aligned_empty(mnb.mnb_packed_size_gidx(w.N, w.K, w.bits, w.bs))
            mnb.mnb_pack_weights_gidx(b, torch.from_numpy(g).cuda(), packed, w.N, w.K, w.bits, w.bs)
            call_flags = flags | mnb.MNB_FLAG_KPERM
        else:
            packed = aligned_empty(mnb.mnb_packed_size(w.N, w.K, w.bits, w.bs))
            mnb.mnb_pack_weights(b, packed, w.N, w.K, w.bits, w.bs)
        del b
        chosen = kernel if kernel != "auto" else mnb.mnb_select_kernel(w.M, w.N, w.K, w.bits, w.bs,
                                                                       w.act_dtype, acc)
        if act_order:
            chosen = "gemv_ks_kperm" if w.M <= 8 else "gather_kperm+gemm_tc"
        ws_bytes = mnb.mnb_workspace_size_ex(w.M, w.N, w.K, w.bits, w.bs, acc, call_flags)
        ws = aligned_empty(ws_bytes) if ws_bytes else None
        # weight copies so that each step streams from HBM
        l2 = torch.cuda.get_device_properties(local).L2_cache_size
        wbytes = packed.numel() + s0.numel() * s0.element_size() + (zp0.numel() if zp0 is not None else 0)
        R = max(2, math.ceil(3 * l2 / wbytes))
        copies = [(packed, s0, zp0)]
        for _ in range(R - 1):
            pb = aligned_empty(packed.numel())
            pb.copy_(packed)
            copies.append((pb, s0.clone(), None if zp0 is None else zp0.clone()))
        yb = torch.empty((w.M, w.N), dtype=TORCH_DT[w.out_dtype], device="cuda")
        stream = torch.cuda.Stream()

        def call(i):
            pb, s, zp = copies[i % R]
            mnb.mnb_matmul_ex(x, pb, s, zp, yb, w.M, w.N, w.K, w.bits, w.bs, w.act_dtype, w.out_dtype,
                              w.scale_dtype, kernel=kernel, stream=stream, flags=call_flags, accuracy_level=acc,
                              workspace=ws)

        t, ck = replay_timed(call, steps, warmup, stream)
        unit, per_step = metric_of(w)
        if act_order and unit == "GB/s":
            per_step += 4 * w.K / 1e9  # the stored permutation, read once per call
        value = whole_job_value(world, steps, per_step, t)
        per_launch_s = t / steps
        # accuracy level 4: activation quantisation + product, except at M <= 4 with 32 <= bs <= 256, where
        # the decode GEMV quantises X itself
        kernels_per_step = 2 if acc == 4 and not (w.M <= 4 and 32 <= w.bs <= 256) else 1
        if act_order and w.M > 8:
            kernels_per_step = 2  # the gather of X into the pack's depth order, then the GEMM
        out = {"workload": w.name, "value": value, "unit": unit, "steps": steps, "ms_per_step": per_launch_s * 1e3,
               "kernel": chosen, "clocks": ck, "weight_copies": R, "launches": steps * kernels_per_step}
        if unit == "GB/s":
            peak = pk["hbm_gbs"]
            out["roofline"] = {"bound": "hbm", "achieved": per_step / per_launch_s, "peak": peak, "unit": "GB/s",
                               "frac": per_step / per_launch_s / peak,
                               "traffic": traffic_for(f"{chosen}:{w.name}" + (":acc4" if acc == 4 else "")),
                               "algorithmic_bytes": w.algorithmic_bytes() + (4 * w.K if act_order else 0),
                               "peak_source": f"{pk_src} hbm_gbs"}
        else:
            peak = pk["bf16_tflops"]
            out["roofline"] = {"bound": "tensor", "achieved": per_step / per_launch_s, "peak": peak,
                               "unit": "TFLOP/s", "frac": per_step / per_launch_s / peak,
                               "traffic": traffic_for(f"{chosen}:{w.name}" + (":acc4" if acc == 4 else "")),
                               "algorithmic_bytes": w.algorithmic_bytes(), "flops": w.flops(),
                               "peak_source": f"{pk_src} bf16_tflops (burst)"}
        if want_e2e:
            # End to end through the C ABI with HOST buffers: X is read from pinned host memory and Y is
            # written to pinned host memory by the library's own kernels (mnb_matmul_host_io), every step.
            xh = x.cpu().pin_memory()
            yh = torch.empty((w.M, w.N), dtype=TORCH_DT[w.out_dtype]).pin_memory()

            def call_host(i):
                pb, s, zp = copies[i % R]
                mnb.mnb_matmul_host_io(xh, pb, s, zp, yh, w.M, w.N, w.K, w.bits, w.bs, w.act_dtype,
                                       w.out_dtype, w.scale_dtype, kernel=kernel, stream=stream, flags=flags,
                                       accuracy_level=acc, workspace=ws)

            te, cke = replay_timed(call_host, steps, warmup, stream)
            out["e2e"] = {"value": whole_job_value(world, steps, per_step, te), "unit": unit,
                          "h2d_bytes_per_step": x.numel() * x.element_size(),
                          "d2h_bytes_per_step": yb.numel() * yb.element_size(),
                          "ms_per_step": te / steps * 1e3, "clocks": cke,
                          "mode": "CUDA graph of mnb_matmul_host_io per step: X read from pinned host memory, "
                                  "Y written to pinned host memory, both by the library's kernels"}
            out["e2e_launches"] = steps * (kernels_per_step + 1)  # + the X fetch kernel
        return out, data

    def measure_moe(w: wl.MoeWorkload, steps: int, warmup: int):
        """The grouped (mixture-of-experts) decode GEMV: one launch over all experts per step."""
        d = wl.generate_moe(w)
        x = to_dev(d["x"], w.act_dtype)
        ids = torch.from_numpy(d["ids"]).cuda()
        ps = mnb.mnb_packed_size(w.N, w.K, w.bits, w.bs)
        packed = aligned_empty(w.E * ps)
        for e in range(w.E):
            be = torch.from_numpy(np.ascontiguousarray(d["b"][e])).cuda()
            mnb.mnb_pack_weights(be, packed[e * ps:(e + 1) * ps], w.N, w.K, w.bits, w.bs)
            del be
        s0 = to_dev(d["scales"], w.scale_dtype)
        zp0 = None if d["zp"] is None else torch.from_numpy(np.ascontiguousarray(d["zp"])).cuda()
        step_bytes = w.bytes(d["ids"])
        l2 = torch.cuda.get_device_properties(local).L2_cache_size
        R = max(2, math.ceil(3 * l2 / step_bytes))
        copies = [(packed, s0, zp0)]
        for _ in range(R - 1):
            pb = aligned_empty(packed.numel())
            pb.copy_(packed)
            copies.append((pb, s0.clone(), None if zp0 is None else zp0.clone()))
        y = torch.empty((w.T, w.S, w.N), dtype=TORCH_DT[w.out_dtype], device="cuda")
        stream = torch.cuda.Stream()

        def call(i):
            pb, s, zp = copies[i % R]
            mnb.mnb_matmul_grouped(x, ids, pb, s, zp, y, w.T, w.S, w.E, w.N, w.K, w.bits, w.bs, w.act_dtype,
                                   w.out_dtype, w.scale_dtype, x_per_slot=w.x_per_slot, stream=stream)

        t, ck = replay_timed(call, steps, warmup, stream)
        per_step = step_bytes / 1e9
        per_launch_s = t / steps
        achieved = per_step / per_launch_s
        return {"workload": w.name, "value": whole_job_value(world, steps, per_step, t), "unit": "GB/s",
                "kernel": "gemv_ks (grouped: pairs <= 8)", "ms_per_step": per_launch_s * 1e3, "steps": steps,
                "experts_active": int(len(np.unique(d["ids"]))), "experts": w.E, "tokens": w.T, "top_k": w.S,
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                             "frac": achieved / pk["hbm_gbs"], "traffic": traffic_for(f"gemv_ks_moe:{w.name}"),
                             "algorithmic_bytes": step_bytes, "peak_source": f"{pk_src} hbm_gbs"},
                "clocks": ck, "weight_copies": R}, steps

    def measure_fp(fmt: int, M: int, N: int, K: int, steps: int, warmup: int):
        """FP8 (E4M3, f32 column scales) or NVFP4 (E4M3 block scales x global) weights, bf16 X and Y:
        native-format bytes (codes, scales, X, Y) per step."""
        rng = np.random.default_rng(wl.SEED_BASE + 50 + fmt)
        act, out = wl.BF16, wl.BF16
        if fmt == mnb.MNB_WF_NVFP4:
            kb = -(-K // 16)
            codes = rng.integers(0, 256, size=(K * N + 1) // 2).astype(np.uint8)
            sc = torch.from_numpy(rng.choice([c for c in range(0x08, 0x40)], size=(kb, N)).astype(np.uint8)).cuda()
            name, wbytes, sbytes = f"decode_m{M}_k{K}_n{N}_nvfp4_bf16", (K * N + 1) // 2, kb * N
        else:
            codes = rng.choice([c for c in range(256) if (c >> 3) & 15 != 15], size=K * N).astype(np.uint8)
            sc = torch.from_numpy(rng.uniform(1e-3, 1e-2, size=N).astype(np.float32)).cuda()
            name, wbytes, sbytes = f"decode_m{M}_k{K}_n{N}_fp8e4m3_bf16", K * N, 4 * N
        wdev = torch.from_numpy(codes).cuda()
        packed = aligned_empty(mnb.mnb_fp_packed_size(N, K, fmt))
        mnb.mnb_pack_fp_weights(wdev, packed, N, K, fmt)
        del wdev
        x = to_dev(wl.to_storage(rng.standard_normal((M, K)), act), act)
        yb = torch.empty((M, N), dtype=TORCH_DT[out], device="cuda")
        l2 = torch.cuda.get_device_properties(local).L2_cache_size
        R = max(2, math.ceil(3 * l2 / (packed.numel() + sbytes)))
        copies = [(packed, sc)]
        for _ in range(R - 1):
            pb = aligned_empty(packed.numel())
            pb.copy_(packed)
            copies.append((pb, sc.clone()))
        stream = torch.cuda.Stream()

        def call(i):
            pb, s = copies[i % R]
            mnb.mnb_matmul_fp(x, pb, s, 0.05, yb, M, N, K, fmt, act, out, stream=stream, flags=flags)

        t, ck = replay_timed(call, steps, warmup, stream)
        # NVFP4 decodes on the tensor-core GEMV unless MNB_FP_KERNEL picks another
        fpk = os.environ.get("MNB_FP_KERNEL", "")
        kern = "fp_generic" if fpk == "generic" else "gemv_nv" if fmt == mnb.MNB_WF_NVFP4 and fpk != "lut" else "gemv_fp"
        per_step = (wbytes + sbytes + M * K * 2 + M * N * 2) / 1e9
        per_launch_s = t / steps
        achieved = per_step / per_launch_s
        return {"workload": name, "value": whole_job_value(world, steps, per_step, t), "unit": "GB/s",
                "kernel": kern, "ms_per_step": per_launch_s * 1e3, "steps": steps,
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                             "frac": achieved / pk["hbm_gbs"], "traffic": traffic_for(f"{kern}:{name}"),
                             "algorithmic_bytes": int(per_step * 1e9), "peak_source": f"{pk_src} hbm_gbs"},
                "clocks": ck, "weight_copies": R}, steps

    w = wl.config(args.config)
    if args.only:
        if args.only == "moe":
            obj, n = measure_moe(wl.MOE_CONFIGS[0], args.steps, args.warmup)
        elif args.only in ("act_order", "act_order_m512"):
            wk = wl.config(1 if args.only == "act_order" else 4)
            sec, _ = measure(wk, args.steps, args.warmup, "auto", False, 0, act_order=True)
            obj, n = {k: sec[k] for k in ("workload", "value", "unit", "kernel", "steps", "ms_per_step", "roofline",
                                          "clocks")}, sec["launches"]
        else:
            obj, n = measure_fp(mnb.MNB_WF_E4M3 if args.only == "fp8" else mnb.MNB_WF_NVFP4, 1, 11008, 4096,
                                args.steps, args.warmup)
        if rank == 0:
            print(json.dumps({"only": args.only, args.only: obj, "gpu_launches": n}), flush=True)
        return
    main, data = measure(w, args.steps, args.warmup, args.kernel, True, args.accuracy_level)
    res = {
        "metric": "int4 MatMulNBits GB/s at M=1, TFLOP/s at M=512; % of roofline",
        "value": main["value"], "unit": main["unit"], "n_gpus": world, "steps": main["steps"],
        "warmup": args.warmup, "ms_per_step": main["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 accumulate (int%d weights, %s activations)" % (w.bits, wl.DTYPE_NAMES[w.act_dtype]),
        "data": "synthetic (seeded, LLM-projection shaped; no trained weights)",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "bits": w.bits, "block_size": w.bs,
                   "zero_points": w.zp is not None, "kernel": main["kernel"],
                   "accuracy_level": args.accuracy_level,
                   "l2": f"inputs larger than L2: {main['weight_copies']} rotating weight copies (>= 3 x L2)",
                   "launch": "CUDA graphs holding all timed steps (one kernel node per step), queued behind a "
                             "GPU spin so the timed region holds device time only"},
        "roofline": main["roofline"], "clocks": main["clocks"], "e2e": main["e2e"],
        "gpu_launches": main["launches"] + main.get("e2e_launches", 0),
    }

    def secondary(key, wk, steps, warmup, acc=0, extra=None, act_order=False):
        sec, _ = measure(wk, steps, warmup, "auto", False, acc, act_order=act_order)
        obj = {"workload": wk.name, "value": sec["value"], "unit": sec["unit"], "kernel": sec["kernel"],
               "steps": sec["steps"], "ms_per_step": sec["ms_per_step"], "roofline": sec["roofline"],
               "clocks": sec["clocks"]}
        obj.update(extra or {})
        res[key] = obj
        res["gpu_launches"] += sec["launches"]

    if args.config == 1 and args.accuracy_level == 0 and not args.no_secondary:
        sw = max(3, args.warmup // 4)
        secondary("m512", wl.config(4), max(20, args.steps // 20), max(3, args.warmup // 20))
        secondary("int8_k11008", wl.config(2), max(20, args.steps // 2), sw)
        secondary("int2_m8", wl.config(3), max(20, args.steps // 2), sw)
        secondary("a8", w, max(20, args.steps // 4), sw, acc=4,
                  extra={"accuracy_level": 4, "launches_per_step": 1})
        secondary("a8_m512", wl.config(4), max(20, args.steps // 20), max(3, args.warmup // 20), acc=4,
                  extra={"accuracy_level": 4, "launches_per_step": 2})
        secondary("act_order", w, max(20, args.steps // 4), sw, act_order=True,
                  extra={"g_idx": "act-order (a seeded permutation of the depths in blocks), MNB_FLAG_KPERM"})
        secondary("act_order_m512", wl.config(4), max(20, args.steps // 20), max(3, args.warmup // 20),
                  act_order=True, extra={"g_idx": "act-order, MNB_FLAG_KPERM: X gathered into the pack's order, "
                                                  "then the prefill GEMM", "launches_per_step": 2})
        moe, n = measure_moe(wl.MOE_CONFIGS[0], max(20, args.steps // 10), max(3, args.warmup // 10))
        res["moe"] = moe
        res["gpu_launches"] += n
        for key, fmt in (("fp8", mnb.MNB_WF_E4M3), ("nvfp4", mnb.MNB_WF_NVFP4)):
            fo, n = measure_fp(fmt, 1, 11008, 4096, max(20, args.steps // 10), sw)
            res[key] = fo
            res["gpu_launches"] += n
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample = cpu_oracle_rate(w, data, args.cpu_seconds)
        res["cpu_baseline"] = {"value": v, "unit": main["unit"], "cores": cores, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_reference(args):
    """The CPU oracle as it stands, on rank 0 only (other ranks exit without work)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    w = wl.config(args.config)
    data = wl.generate(w)
    unit, _ = metric_of(w)
    per = max(0.5, min(10.0, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_oracle_rate(w, data, per)
    vals = []
    t0 = time.perf_counter()
    cores, sample = None, None
    for _ in range(args.steps):
        v, cores, sample = cpu_oracle_rate(w, data, per)
        vals.append(v)
    wall = time.perf_counter() - t0
    value = statistics.median(vals)
    res = {"impl": "reference", "metric": "int4 MatMulNBits GB/s at M=1, TFLOP/s at M=512; % of roofline",
           "value": value, "unit": unit, "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": wall / max(1, args.steps) * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64 (CPU oracle)", "data": "synthetic (seeded)",
           "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "bits": w.bits, "block_size": w.bs},
           "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                            "sample": f"per step: {sample}"},
           "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)
    return res


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)
