#!/usr/bin/env python3
"""Benchmark of the AdaComp hot path on GB300: compress + decode-accumulate.

One step = one pass of the whole path over one batch of synthetic gradients: every
learner compresses every layer of the workload (fused streaming kernel, scale,
codes and fix-up), the message lengths are read back (what an exchange of the
variable-length messages would carry), and all learners' messages are decoded and
accumulated into dense gradients. The default workload is the aggregation
configuration: 16 learners, each with its own carried residue and N(0, 1e-3) dW
over one flat 10^8-element fp32 layer at L_T = 500, and one decode of all 16
messages. ``--workload resnet50 | lstm_fc | gpt1p3b | fc400k`` runs the other
gradient sets with one learner (``gpt1p3b`` at ``--bin-len`` 50, 500 or 5000).

The JSON line reports gradient elements/s (value), algorithmic HBM GB/s and their
fraction of the measured copy bandwidth, the dominant kernel's roofline, an
end-to-end figure through the C ABI with host buffers, and the oracle timed on
host cores. ``--impl reference`` times the oracle alone (this build's reference
arm). With torchrun and N > 1 every rank runs an independent replica.
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
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from residual_gradient_compression_gb300 import workloads as wl  # noqa: E402

METRIC = "gradient elements/s and HBM GB/s (% of GB300 roofline) for compress+decode"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # the GB300's nominal HBM3e bandwidth


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["adacomp", "reference"], default="adacomp")
    p.add_argument("--workload", default="flat100m",
                   choices=["resnet50", "fc400k", "lstm_fc", "gpt1p3b", "flat100m"])
    p.add_argument("--bin-len", type=int, default=500, help="L_T for gpt1p3b")
    p.add_argument("--streams", type=int, default=3, choices=[1, 2, 3, 4],
                   help="learners' compress calls taking turns on this many streams (default three)")
    p.add_argument("--layers", type=int, default=0,
                   help="only the first N layers of the workload (a smaller case, for profiling)")
    p.add_argument("--learners", type=int, default=16, help="K for flat100m")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle sample budget")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-lazy", action="store_true", help="skip the deferred fix-up measurement")
    p.add_argument("--no-sgd", action="store_true", help="skip the fused decode + SGD measurement")
    p.add_argument("--min-timed-seconds", type=float, default=1.5,
                   help="repeat the K timed steps until the clock sampler has covered this long")
    p.add_argument("--residue-contrast", action="store_true",
                   help="instead of the benchmark: residue range and compression per carried step of AdaComp "
                        "and of Local Selection on one 4096x4096 layer at L_T 50, 500 and 5000")
    p.add_argument("--contrast-steps", type=int, default=25)
    return p.parse_args()


# ---------------------------------------------------------------- distributed (replicas)
def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value over all ranks (the slowest replica sets the job's time)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- workloads
def workload_layers(args):
    ls = wl.layers("gpt1p3b", args.bin_len) if args.workload == "gpt1p3b" else wl.layers(args.workload)
    return ls[:args.layers] if args.layers else ls


def learners(args):
    return args.learners if args.workload == "flat100m" else 1


def chunks(seq, size):
    return [seq[i:i + size] for i in range(0, len(seq), size)]


def algorithmic_bytes(layers, nnz, K):
    """Minimum bytes each stage of one step must move, summed over the layers.

    nnz: codes per (learner, layer) compress, learner-major (K runs over `layers`).
    stream (the streaming kernel): read residue (4 B) and dW (2 or 4 B) and write
    residue (4 B) per element, and write the per-bin counts (2B);
    post (finalise, codes, fix-up): write the header (8 B) and the codes (w*nnz), and
    rewrite each sent residue (4 B read + 4 B write);
    decode: a layer whose learners together sent at least n/16 codes is streamed
    (read and write every dense element, 8 B); a sparser one is updated in place
    (8 B per code); plus reading the messages, and their counts once more (2B) for
    the scan.
    Returns (stream bytes, post bytes, decode bytes).
    """
    stream = post = dec = 0
    for i, ly in enumerate(layers):
        d = 2 if ly.dw_dtype == "bf16" else 4
        B = -(-ly.numel // ly.bin_len)
        w = 1 if ly.bin_len < 64 else 2
        zs = [nnz[k * len(layers) + i] for k in range(K)]
        stream += K * (ly.numel * (8 + d) + 2 * B)
        post += sum(8 + w * z + 8 * z for z in zs)
        dense = 16 * sum(zs) >= ly.numel
        dec += (8 * ly.numel if dense else 8 * sum(zs)) + sum(8 + 2 * B + w * z for z in zs) + 2 * B * K
    return stream, post, dec


# The source files each profiled kernel is built from (its .cu and the headers it includes).
KERNEL_SOURCES = {
    "slice_kernel": ("compress_sliced.cu", "compress_common.cuh", "adacomp_internal.cuh"),
    "slice_emit_kernel": ("compress_sliced.cu", "compress_common.cuh", "adacomp_internal.cuh"),
    "slice_codes_kernel": ("compress_sliced.cu", "compress_common.cuh", "adacomp_internal.cuh"),
    "block_kernel": ("compress_sliced.cu", "compress_common.cuh", "adacomp_internal.cuh"),
    "compress_kernel": ("compress.cu", "compress_common.cuh", "adacomp_internal.cuh"),
    "accumulate_kernel": ("decode.cu", "adacomp_internal.cuh"),
    "sparse_accumulate_kernel": ("decode.cu", "adacomp_internal.cuh"),
    "check_kernel": ("decode.cu", "adacomp_internal.cuh"),
}


def source_hash(kernel=None):
    """sha256 prefix of a kernel's source files (all of csrc/ when kernel is None)."""
    d = os.path.join(ROOT, "residual_gradient_compression_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel) or sorted(os.listdir(d))
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(d, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_hbm_gbs():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(kernel: str, workload: str, bytes_per_launch: float):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel sources; None otherwise. A summary taken on a smaller case of the
    workload (one whose launch is too large to capture) is scaled to this launch by
    the ratio of algorithmic bytes, the traffic of a streaming kernel growing in
    proportion to the elements it streams."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("source_sha") != source_hash(kernel):
        return None
    dram = rec.get("dram_bytes_per_launch")
    if dram is not None and rec.get("scale_by_algorithmic_bytes"):
        dram *= bytes_per_launch / rec["algorithmic_bytes_per_launch"]
    return dram


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        # the samples go to a temporary file, or to ADACOMP_CLOCKS_CSV when it is set
        self.path = os.environ.get("ADACOMP_CLOCKS_CSV") or os.path.join(
            tempfile.gettempdir(), f"adacomp_clocks_rank{gpu_index}_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path) or ".", exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return None

        def mhz(v):
            try:
                return float(v.split()[0])
            except Exception:
                return float("nan")
        sm = [mhz(r[1]) for r in rows]
        mx = [mhz(r[2]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        good = [x for x in sm if not math.isnan(x)]
        return {"sm_mhz": statistics.median(good) if good else None,
                "sm_max_mhz": max(x for x in mx if not math.isnan(x)) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def _flat_views(total_numels, dtype, device, fill=None, pinned=False):
    """One buffer holding several tensors, each starting on a 16-byte boundary."""
    esz = torch.empty(0, dtype=dtype).element_size()
    per = max(1, 16 // esz)
    offs, cur = [], 0
    for n in total_numels:
        offs.append(cur)
        cur += -(-n // per) * per
    if pinned:
        buf = torch.empty(max(cur, 1), dtype=dtype, pin_memory=True)
    else:
        buf = torch.zeros(max(cur, 1), dtype=dtype, device=device)
    return buf, [buf[o:o + n] for o, n in zip(offs, total_numels)]


class DeviceRun:
    """All device buffers and prepared C-ABI calls of one replica."""

    def __init__(self, args, layers, dev):
        import ctypes
        import residual_gradient_compression_gb300 as ac
        from residual_gradient_compression_gb300 import build
        build.build()
        self.ac, self.ct, self.L = ac, ctypes, ac.lib()
        self.args, self.layers, self.dev = args, layers, dev
        self.K = learners(args)
        self.sets = 4 if args.workload in ("resnet50", "fc400k", "lstm_fc") else 2
        names = [l.name for l in wl.layers(args.workload, args.bin_len if args.workload == "gpt1p3b" else None)]
        self.gidx = chunks(list(range(len(layers))), ac.MAX_GROUP)
        self.h = [ac.adacomp_init_group([layers[i].numel for i in g], [layers[i].bin_len for i in g],
                                        [ac.BF16 if layers[i].dw_dtype == "bf16" else ac.F32 for i in g])
                  for g in self.gidx]
        numels = [l.numel for l in layers]
        bf16 = layers[0].dw_dtype == "bf16"
        self.dw_dtype = torch.bfloat16 if bf16 else torch.float32
        # residue per learner, dense per layer, dW sets per learner
        self.res = [_flat_views(numels, torch.float32, dev) for _ in range(self.K)]
        self.dense = _flat_views(numels, torch.float32, dev)
        self.dw = []
        for k in range(self.K):
            per_set = []
            for s in range(self.sets):
                buf, views = _flat_views(numels, self.dw_dtype, dev)
                for i, ly in enumerate(layers):
                    views[i].copy_(wl.gen_dw(args.workload, names.index(ly.name), ly, s, learner=k, device=dev))
                per_set.append((buf, views))
            self.dw.append(per_set)
        maxmsg = [m for h in self.h for m in h.max_msg_bytes]
        self.msg = [_flat_views(maxmsg, torch.uint8, dev) for _ in range(self.K)]
        self.dws_bytes = [h.decode_ws_bytes(self.K) for h in self.h]
        self.dec_ws = [torch.zeros(b, dtype=torch.uint8, device=dev) for b in self.dws_bytes]
        self.ring = max(1, args.steps)
        self.ws = [[[torch.zeros(h.compress_ws_bytes, dtype=torch.uint8, device=dev) for h in self.h]
                    for _ in range(self.K)] for _ in range(self.ring)]
        self._prepare()

    def _prepare(self):
        ct, VP = self.ct, self.ct.c_void_p
        self.c_res, self.c_msg, self.c_cap, self.c_dw = [], [], [], []
        for k in range(self.K):
            r, m, c = [], [], []
            for g in self.gidx:
                r.append((VP * len(g))(*[self.res[k][1][i].data_ptr() for i in g]))
                m.append((VP * len(g))(*[self.msg[k][1][i].data_ptr() for i in g]))
                c.append((ct.c_size_t * len(g))(*[self.msg[k][1][i].numel() for i in g]))
            self.c_res.append(r)
            self.c_msg.append(m)
            self.c_cap.append(c)
            self.c_dw.append([[(VP * len(g))(*[self.dw[k][s][1][i].data_ptr() for i in g]) for g in self.gidx]
                              for s in range(self.sets)])
        self.c_dec_msgs = [(VP * (len(g) * self.K))(*[self.msg[k][1][i].data_ptr() for i in g
                                                        for k in range(self.K)]) for g in self.gidx]
        self.msg_sets = [(self.msg, self.c_msg, self.c_dec_msgs)]
        self.c_dense = [(VP * len(g))(*[self.dense[1][i].data_ptr() for i in g]) for g in self.gidx]

    def add_msg_set(self):
        """A second set of message buffers (and their pointer arrays), so that one
        step's messages can be copied to the host while the next step writes its own."""
        VP = self.ct.c_void_p
        maxmsg = [m for h in self.h for m in h.max_msg_bytes]
        msg = [_flat_views(maxmsg, torch.uint8, self.dev) for _ in range(self.K)]
        c_msg = [[(VP * len(g))(*[msg[k][1][i].data_ptr() for i in g]) for g in self.gidx] for k in range(self.K)]
        c_dec = [(VP * (len(g) * self.K))(*[msg[k][1][i].data_ptr() for i in g for k in range(self.K)])
                 for g in self.gidx]
        self.msg_sets.append((msg, c_msg, c_dec))

    def launches_per_step(self):
        # compress: streaming kernel, finalise, codes + fix-up; decode: sums, scan, validation,
        # accumulate (staged and in place)
        return self.K * len(self.gidx) * 3 + len(self.gidx) * 5

    RESULT_AT = 2064  # offset of a layer's result {s, status, nnz, msg_bytes} in its 2112-byte block

    def _host_results(self):
        if not hasattr(self, "host_res"):
            self.res_bytes = [64 + 2112 * len(g) for g in self.gidx]
            # one pinned buffer per group, a row per learner; numpy views made once
            self.host_buf = [torch.empty((self.K, rb), dtype=torch.uint8, pin_memory=True) for rb in self.res_bytes]
            self.host_np = [b.numpy() for b in self.host_buf]
            self.host_res = [[self.host_buf[gi][k] for gi in range(len(self.gidx))] for k in range(self.K)]
        return self.host_res

    def message_lengths(self, ws_of):
        """Reads every (learner, group) results area back to the host (one copy each,
        then one wait on the stream) and returns, per group, the layer-major array
        of message lengths the decode takes; raises on a device status."""
        host = self._host_results()
        for k in range(self.K):
            for gi in range(len(self.gidx)):
                host[k][gi].copy_(ws_of(k, gi)[:self.res_bytes[gi]], non_blocking=True)
        torch.cuda.current_stream().synchronize()
        if not hasattr(self, "len_bufs"):
            self.len_bufs = [np.zeros(len(g) * self.K, np.uint64) for g in self.gidx]
            self.len_ptrs = [b.ctypes.data_as(self.ct.POINTER(self.ct.c_uint64)) for b in self.len_bufs]
        ra = self.RESULT_AT
        for gi, g in enumerate(self.gidx):
            nl = len(g)
            # every learner's layer blocks (2112 bytes after the 64-byte control block);
            # in each, the result {s f32, status u32, nnz u64, msg_bytes u64} at RESULT_AT
            blk = self.host_np[gi][:, 64:64 + 2112 * nl].reshape(self.K, nl, 2112)
            status = blk[:, :, ra + 4:ra + 8].copy().view(np.uint32)
            if status.any():
                raise RuntimeError(f"device status {int(status[status != 0][0])}")
            mb = blk[:, :, ra + 16:ra + 24].copy().view(np.uint64)[:, :, 0]  # (K, layers)
            self.len_bufs[gi][:] = mb.T.ravel()  # layer-major: [layer * K + learner]
        return self.len_ptrs

    def step(self, i, stream_ptr, k1_events=None, dec_events=None, ws_fixed=None, msg_set=0):
        """One step: every learner's compress, the message lengths read back (the
        exchange of variable-length messages would carry them), then the decode of
        the step's messages. ws_fixed: one workspace per (learner, group) used by
        every step (a deferred fix-up keeps its pending corrections there), instead of
        the per-step ring."""
        L, s = self.L, i % self.sets
        _, c_msg, c_dec_msgs = self.msg_sets[msg_set]

        def ws_of(k, gi):
            return ws_fixed[k][gi] if ws_fixed is not None else self.ws[i % self.ring][k][gi]

        # the compress calls (learner by learner, launch group by launch group) take turns
        # on the launch stream and args.streams - 1 side streams, so that one call's
        # short launches (finalise, codes) overlap the next one's streaming kernel; the
        # side streams start after everything before the step and the lengths are read
        # once all are done
        nstreams = self.args.streams if self.K * len(self.h) > 1 else 1
        if nstreams > 1:
            if len(getattr(self, "sides", [])) < nstreams - 1:
                self.sides = [torch.cuda.Stream() for _ in range(nstreams - 1)]
                self.side_ptrs = [self.ct.c_void_p(x.cuda_stream) for x in self.sides]
            for x in self.sides[:nstreams - 1]:
                x.wait_stream(torch.cuda.current_stream())
        for k in range(self.K):
            for gi, h in enumerate(self.h):
                turn = (k * len(self.h) + gi) % nstreams
                sptr = self.side_ptrs[turn - 1] if turn else stream_ptr
                if k1_events is not None:
                    e = k1_events[k * len(self.h) + gi]
                    L.adacomp_set_timing_events(h.ptr, self.ct.c_void_p(e[0].cuda_event),
                                                self.ct.c_void_p(e[1].cuda_event),
                                                self.ct.c_void_p(e[2].cuda_event))
                ws = ws_of(k, gi)
                st = L.adacomp_compress_group(h.ptr, self.c_res[k][gi], self.c_dw[k][s][gi], c_msg[k][gi],
                                              self.c_cap[k][gi], ws.data_ptr(), ws.numel(), sptr)
                if st:
                    raise RuntimeError(f"adacomp_compress_group: {st}")
        if nstreams > 1:
            for x in self.sides[:nstreams - 1]:
                torch.cuda.current_stream().wait_stream(x)
        lens = self.message_lengths(ws_of)
        if dec_events is not None:
            dec_events[0].record()
        for gi, h in enumerate(self.h):
            st = L.adacomp_decode_accumulate_group(h.ptr, c_dec_msgs[gi], lens[gi], self.K, self.c_dense[gi],
                                                   self.dec_ws[gi].data_ptr(), self.dec_ws[gi].numel(),
                                                   stream_ptr)
            if st:
                raise RuntimeError(f"adacomp_decode_accumulate_group: {st}")
        if dec_events is not None:
            dec_events[1].record()
        return lens

    def clear_timing(self):
        for h in self.h:
            self.L.adacomp_set_timing_events(h.ptr, None, None, None)

    def step_results(self, i):
        """[(nnz, msg_bytes, status)] per learner per layer for ring slot i."""
        out = []
        for k in range(self.K):
            for gi, (h, g) in enumerate(zip(self.h, self.gidx)):
                ws = self.ws[i % self.ring][k][gi]
                blk = ws[64:64 + 2112 * len(g)].cpu().numpy()
                for j in range(len(g)):
                    o = 2112 * j + self.RESULT_AT
                    status = int(blk[o + 4:o + 8].view(np.uint32)[0])
                    nnz = int(blk[o + 8:o + 16].view(np.uint64)[0])
                    mb = int(blk[o + 16:o + 24].view(np.uint64)[0])
                    out.append((nnz, mb, status))
        return out


def _new_events(n):
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record()  # creates the underlying CUDA event
    return evs


def bench_config(args, layers, K, world):
    """The workload description both arms print (the reference arm the same dict)."""
    return {"workload": args.workload, "layers": len(layers),
            "elements_per_learner": sum(l.numel for l in layers), "learners": K,
            "bin_len": sorted({l.bin_len for l in layers}),
            "dw_dtype": layers[0].dw_dtype, "residue_dtype": "f32",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "compress_streams": args.streams if K * (-(-len(layers) // 128)) > 1 else 1,
            "l2": "inputs larger than L2 (dW rotates over %d sets)" % (
                4 if args.workload in ("resnet50", "fc400k", "lstm_fc") else 2)}


def residue_range(run):
    """min and max of every learner's residue after the last step (eager fix-up)."""
    lo, hi = math.inf, -math.inf
    for k in range(run.K):
        mn, mx = torch.aminmax(run.res[k][0])
        lo, hi = min(lo, float(mn)), max(hi, float(mx))
    return [lo, hi]


def launch_times(args, run, sp, step_no):
    """Per-launch times of the streaming kernel and of the finalise + codes launches,
    each kernel alone: the same steps on one stream with events recorded around every
    launch (one repetition after a step of warm-up). Returns the repetition's step
    time and the two lists."""
    saved = args.streams
    args.streams = 1
    try:
        ncalls = run.K * len(run.h)
        k1_events = [[_new_events(3) for _ in range(ncalls)] for _ in range(args.steps)]
        run.last_lens = run.step(step_no, sp)
        start, end = _new_events(2)
        torch.cuda.synchronize()
        start.record()
        for i in range(args.steps):
            run.last_lens = run.step(step_no + 1 + i, sp, k1_events[i])
        end.record()
        torch.cuda.synchronize()
        run.clear_timing()
        for i in range(args.steps):
            for r in run.step_results(step_no + 1 + i):
                if r[2] != 0:
                    raise RuntimeError(f"device status {r[2]} in the one-stream steps")
        k1 = [e[0].elapsed_time(e[1]) for st in k1_events for e in st]
        fx = [e[1].elapsed_time(e[2]) for st in k1_events for e in st]
        return start.elapsed_time(end), k1, fx
    finally:
        args.streams = saved


def run_device(args, rank, world):
    dev = torch.device("cuda", torch.cuda.current_device())
    layers = workload_layers(args)
    run = DeviceRun(args, layers, dev)
    stream = torch.cuda.current_stream()
    sp = run.ct.c_void_p(stream.cuda_stream)
    n_elems = sum(l.numel for l in layers) * run.K

    for i in range(args.warmup):
        run.step(i, sp)
    torch.cuda.synchronize()
    for i in range(args.warmup):  # warm-up results must be clean
        for nnz, mb, st in run.step_results(i):
            if st != 0:
                raise RuntimeError(f"device status {st} during warm-up")

    dec_events = [_new_events(2) for _ in range(args.steps)]
    start, end = _new_events(2)
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    reps, t0 = [], time.perf_counter()
    step_no = args.warmup
    while True:
        barrier(world)
        torch.cuda.synchronize()
        start.record()
        for i in range(args.steps):
            run.last_lens = run.step(step_no + i, sp, None, dec_events[i])
        end.record()
        torch.cuda.synchronize()
        barrier(world)
        ms = start.elapsed_time(end)
        dec = [e[0].elapsed_time(e[1]) for e in dec_events]
        res = [run.step_results(step_no + i) for i in range(args.steps)]
        reps.append((ms, dec, res))
        step_no += args.steps
        if time.perf_counter() - t0 >= args.min_timed_seconds or len(reps) >= 500:
            break
    clocks = sampler.stop() if sampler else None
    rrange = residue_range(run)
    # each kernel's launch time alone: the same steps on one stream, events on every launch
    one_ms, k1, fx = launch_times(args, run, sp, step_no)

    # the median repetition is reported
    order = sorted(range(len(reps)), key=lambda r: reps[r][0])
    ms, dec, res = reps[order[len(order) // 2]]
    ms = max_over_ranks(ms, world)
    for step_res in res:
        for nnz, mb, st in step_res:
            if st != 0:
                raise RuntimeError(f"device status {st} in the timed region")
    lay_k = [ly for _ in range(run.K) for ly in layers]
    per_step = [algorithmic_bytes(layers, [r[0] for r in step_res], run.K) for step_res in res]
    k1_bytes = sum(p[0] for p in per_step)
    fix_bytes = sum(p[1] for p in per_step)
    dec_bytes = sum(p[2] for p in per_step)
    total_bytes = k1_bytes + fix_bytes + dec_bytes
    msg_bytes = sum(r[1] for step_res in res for r in step_res)
    nnz_total = sum(r[0] for step_res in res for r in step_res)
    bins_total = sum(-(-ly.numel // ly.bin_len) for ly in lay_k) * args.steps

    peak, peak_kind = measured_hbm_gbs()
    # the streaming kernel of the launch: warp-sliced when every bin length is 16..509,
    # block-sliced when every one is 510..8189, else the look-back kernel
    if all(16 <= ly.bin_len <= 509 for ly in layers):
        stream_kernel = "slice_kernel"
    elif all(510 <= ly.bin_len <= 8189 for ly in layers):
        stream_kernel = "block_kernel"
    else:
        stream_kernel = "compress_kernel"
    k1_ms_per_launch = statistics.mean(k1)
    k1_bytes_per_launch = k1_bytes / (args.steps * run.K * len(run.h))
    achieved = k1_bytes_per_launch / (k1_ms_per_launch * 1e-3) / 1e9
    step_gbs = total_bytes / (ms * 1e-3) / 1e9
    dec_gbs = dec_bytes / args.steps / (statistics.mean(dec) * 1e-3) / 1e9
    value = n_elems * args.steps * world / (ms * 1e-3)

    out = {
        "metric": METRIC, "value": value, "unit": "elements/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32" if run.dw_dtype == torch.float32 else "bf16+f32",
        "data": "synthetic",
        "config": bench_config(args, layers, run.K, world),
        "timed_repetitions": len(reps),
        "hbm_gbs": step_gbs, "hbm_frac": step_gbs / peak, "hbm_peak_gbs": peak, "hbm_peak_kind": peak_kind,
        "hbm_frac_nominal": step_gbs / NOMINAL_HBM_GBS, "hbm_nominal_gbs": NOMINAL_HBM_GBS,
        "compress_ms_per_step": (sum(k1) + sum(fx)) / args.steps, "decode_ms_per_step": statistics.mean(dec),
        "decode_gbs": dec_gbs, "decode_frac": dec_gbs / peak,
        "stream_ms_per_launch": k1_ms_per_launch,
        "finalize_emit_ms_per_launch": statistics.mean(fx),
        "compression_ratio": 4.0 * n_elems * args.steps / msg_bytes,
        "message_bytes_per_learner": msg_bytes / args.steps / run.K,
        "sent_per_bin": nnz_total / bins_total,
        "residue_range": rrange,
        "roofline": {"kernel": stream_kernel, "bound": "hbm", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "peak_kind": peak_kind,
                     "frac_nominal": achieved / NOMINAL_HBM_GBS,
                     "traffic": profiled_traffic(stream_kernel, args.workload, k1_bytes_per_launch),
                     "bytes_per_launch": k1_bytes_per_launch, "ms_per_launch": k1_ms_per_launch},
        "gpu_launches": run.launches_per_step() * args.steps,
        "clocks": clocks,
    }
    if not args.no_e2e:
        out["e2e"] = run_e2e(args, run, layers, sp, world)
    if not args.no_lazy:
        out["lazy_fixup"] = run_lazy(args, run, sp, world, n_elems)
    if run.K * len(run.h) > 1 and args.streams > 1:  # the same steps with every call on one stream
        out["one_stream"] = {"value": n_elems * args.steps * world / (one_ms * 1e-3), "unit": "elements/s",
                             "ms_per_step": one_ms / args.steps}
    if not args.no_sgd:
        out["decode_sgd"] = run_decode_sgd(args, run, sp, world, layers)
        out["decode_adam"] = run_decode_sgd(args, run, sp, world, layers, adam=True)
    return out, run


def run_decode_sgd(args, run, sp, world, layers, adam=False):
    """The decode fused with one optimiser step on the last timed step's messages:
    momentum SGD (adacomp_decode_sgd_group: weights and momentum read and written
    once, 16 B per element) or Adam (adacomp_decode_adam_group: weights and both
    moments, 24 B per element), instead of a dense sum plus a separate optimiser pass."""
    ct = run.ct
    numels = [l.numel for l in layers]
    bufs = [_flat_views(numels, torch.float32, run.dev) for _ in range(3 if adam else 2)]
    # weights, and optimiser state as it stands some steps into training (nonzero
    # nearly everywhere: every element has received codes in some earlier step)
    bufs[0][0].normal_()
    bufs[1][0].normal_(0.0, 1e-4)
    if adam:
        bufs[2][0].uniform_(1e-9, 1e-8)
    VP = ct.c_void_p
    ptrs = [[(VP * len(g))(*[views[i].data_ptr() for i in g]) for g in run.gidx] for _, views in bufs]
    stream = torch.cuda.current_stream()
    f = ct.c_float
    lr, b1, b2, eps, t = 1e-3, 0.9, 0.999, 1e-8, 10

    def once():
        for gi, h in enumerate(run.h):
            if adam:
                st = run.L.adacomp_decode_adam_group(
                    h.ptr, run.c_dec_msgs[gi], run.last_lens[gi], run.K, ptrs[0][gi], ptrs[1][gi], ptrs[2][gi],
                    f(lr), f(b1), f(b2), f(eps), f(1 - b1 ** t), f(1 - b2 ** t), f(1.0 / run.K),
                    run.dec_ws[gi].data_ptr(), run.dec_ws[gi].numel(), sp)
            else:
                st = run.L.adacomp_decode_sgd_group(h.ptr, run.c_dec_msgs[gi], run.last_lens[gi], run.K, ptrs[0][gi],
                                                    ptrs[1][gi], f(lr), f(0.9), f(1.0 / run.K),
                                                    run.dec_ws[gi].data_ptr(), run.dec_ws[gi].numel(), sp)
            if st:
                raise RuntimeError(f"fused decode: {st}")

    for _ in range(3):
        once()
    start, end = _new_events(2)
    reps, t0 = [], time.perf_counter()
    while True:
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(args.steps):
            once()
        end.record(stream)
        torch.cuda.synchronize()
        reps.append(start.elapsed_time(end) / args.steps)
        if time.perf_counter() - t0 >= args.min_timed_seconds / 3 or len(reps) >= 200:
            break
    for gi, h in enumerate(run.h):
        if run.ac.adacomp_decode_status(h, run.dec_ws[gi]) != run.ac.OK:
            raise RuntimeError("the fused decode rejected a message")
    ms = max_over_ranks(sorted(reps)[len(reps) // 2], world)
    msg_bytes = int(sum(int(b.sum()) for b in run.len_bufs))
    bins = sum(-(-l.numel // l.bin_len) for l in layers) * run.K
    algo = (24 if adam else 16) * sum(numels) + msg_bytes + 2 * bins
    del bufs
    peak, _ = measured_hbm_gbs()
    return {"ms_per_decode": ms, "algorithmic_bytes": algo, "achieved_gbs": algo / (ms * 1e-3) / 1e9,
            "frac": algo / (ms * 1e-3) / 1e9 / peak,
            "optimizer": ("Adam, lr 1e-3, betas (0.9, 0.999), eps 1e-8, step 10, grad_scale 1/K, "
                          "moments m ~ N(0, 1e-4), v ~ U(1e-9, 1e-8)" if adam
                          else "momentum SGD, lr 1e-3, mu 0.9, grad_scale 1/K, momentum ~ N(0, 1e-4)")}


def run_lazy(args, run, sp, world, n_elems):
    """The same steps with the residue fix-up deferred to the next step
    (adacomp_set_lazy_fixup): identical messages, no fix-up kernel for warp-sliced
    layers. Reported beside the eager numbers, not as the headline."""
    ac = run.ac
    for h in run.h:
        ac.adacomp_set_lazy_fixup(h, True)
    ws = [[torch.zeros(h.compress_ws_bytes, dtype=torch.uint8, device=run.dev) for h in run.h]
          for _ in range(run.K)]
    stream = torch.cuda.current_stream()
    for i in range(max(3, args.warmup)):
        run.last_lens = run.step(i, sp, ws_fixed=ws)
    start, end = _new_events(2)
    reps, t0, step_no = [], time.perf_counter(), 0
    while True:
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(args.steps):
            run.last_lens = run.step(step_no + i, sp, ws_fixed=ws)
        end.record(stream)
        torch.cuda.synchronize()
        reps.append(start.elapsed_time(end))
        step_no += args.steps
        if time.perf_counter() - t0 >= args.min_timed_seconds / 2 or len(reps) >= 200:
            break
    ms = max_over_ranks(sorted(reps)[len(reps) // 2], world)
    # one more step with every launch's events: the streaming kernel (which applies
    # the previous call's corrections) and the finalise + codes launches
    ev = [_new_events(3) for _ in range(run.K * len(run.h))]
    saved, args.streams = args.streams, 1  # each kernel alone
    try:
        run.last_lens = run.step(step_no, sp, k1_events=ev, ws_fixed=ws)
        torch.cuda.synchronize()
    finally:
        args.streams = saved
    run.clear_timing()
    k1 = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    fx = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    for k in range(run.K):
        for gi, h in enumerate(run.h):
            for li in range(h.num_layers):
                if ac.adacomp_query(h, ws[k][gi], li)[2] != ac.OK:
                    raise RuntimeError("device status not OK with the deferred fix-up")
            ac.adacomp_materialize_group(h, run.res[k][1][run.gidx[gi][0]:run.gidx[gi][-1] + 1], ws[k][gi])
    for h in run.h:
        ac.adacomp_set_lazy_fixup(h, False)
    torch.cuda.synchronize()
    return {"value": n_elems * args.steps * world / (ms * 1e-3), "unit": "elements/s",
            "ms_per_step": ms / args.steps, "timed_repetitions": len(reps),
            "stream_ms_per_launch": k1, "finalize_codes_ms_per_launch": fx,
            "finalize_codes_share_of_stream": fx / k1}


E2E_REPS = 3


def run_e2e(args, run, layers, sp, world):
    """Same steps through the C ABI with host buffers: each step copies its dW from
    pinned host memory, runs the path (the message lengths come back to the host
    before the decode, as an exchange of the messages would need them), and copies
    the messages back to pinned host memory (runs of neighbouring messages).

    The copies overlap the computation of neighbouring steps: the dW of step i + 1
    goes up on a copy stream (into the dW slot it uses, once the step that last read
    that slot is done) while step i computes, and the messages of step i go down on
    a second copy stream from one of two message buffer sets while step i + 1
    computes into the other. Also reported: the host-to-device rate of the upload
    alone (every learner's dW, one copy each, timed with events on the copy stream)."""
    numels = [l.numel for l in layers]
    host_dw = []
    for k in range(run.K):
        buf, views = _flat_views(numels, run.dw_dtype, "cpu", pinned=True)
        buf.copy_(run.dw[k][0][0][:buf.numel()])
        host_dw.append(buf)
    if len(run.msg_sets) < 2:
        run.add_msg_set()
    host_msg = [torch.empty(run.msg[k][0].numel(), dtype=torch.uint8, pin_memory=True) for k in range(run.K)]
    msg_offs = [[v.data_ptr() - run.msg[k][0].data_ptr() for v in run.msg[k][1]] for k in range(run.K)]
    comp = torch.cuda.current_stream()
    up = torch.cuda.Stream()
    down = torch.cuda.Stream()
    steps = args.steps
    h2d = d2h = 0
    slot_free = [None] * run.sets   # compute of the step that last read each dW slot
    msgs_free = [None, None]        # message copies of the step that last wrote each set
    up_done = {}

    def upload(j):
        nonlocal h2d
        slot = j % run.sets
        if slot_free[slot] is not None:
            up.wait_event(slot_free[slot])
        with torch.cuda.stream(up):
            for k in range(run.K):
                run.dw[k][slot][0][:host_dw[k].numel()].copy_(host_dw[k], non_blocking=True)
                h2d += host_dw[k].numel() * host_dw[k].element_size()
        ev = torch.cuda.Event()
        ev.record(up)
        up_done[j] = ev

    def messages_down(j, lens):
        """Enqueues the message copies of step j (its compress is complete)."""
        nonlocal d2h
        msg = run.msg_sets[j % 2][0]
        with torch.cuda.stream(down):
            for k in range(run.K):
                spans, li = [], 0
                for gi, g in enumerate(run.gidx):
                    for jj in range(len(g)):
                        spans.append((msg_offs[k][li], int(run.len_bufs[gi][jj * run.K + k])))
                        li += 1
                # one copy per run of messages: neighbours whose gap (the unused tail of
                # a buffer sized for the worst case) is under 256 KB share a copy
                runs = []
                for off, ln in sorted(spans):
                    if runs and off - runs[-1][1] < (256 << 10):
                        runs[-1][1] = off + ln
                    else:
                        runs.append([off, off + ln])
                for r0, r1 in runs:
                    host_msg[k][r0:r1].copy_(msg[k][0][r0:r1], non_blocking=True)
                    d2h += r1 - r0
        ev = torch.cuda.Event()
        ev.record(down)
        msgs_free[j % 2] = ev

    def timed_steps():
        upload(0)
        for i in range(steps):
            if i + 1 < steps:
                upload(i + 1)
            comp.wait_event(up_done.pop(i))
            if msgs_free[i % 2] is not None:
                comp.wait_event(msgs_free[i % 2])
            lens = run.step(i, sp, msg_set=i % 2)
            done = torch.cuda.Event()
            done.record(comp)
            slot_free[i % run.sets] = done
            messages_down(i, lens)
        torch.cuda.synchronize()

    # the host link is shared with the machine's other work, so its rate varies from
    # moment to moment: the median of E2E_REPS repetitions of the timed steps is reported
    rep_secs = []
    for _ in range(E2E_REPS):
        h2d = d2h = 0
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        timed_steps()
        rep_secs.append(max_over_ranks(time.perf_counter() - t0, world))
        d2h += steps * run.K * sum(run.res_bytes)
    secs = sorted(rep_secs)[len(rep_secs) // 2]
    n_elems = sum(numels) * run.K

    # the upload alone
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(up):
        e0.record(up)
        nb = 0
        for k in range(run.K):
            run.dw[k][0][0][:host_dw[k].numel()].copy_(host_dw[k], non_blocking=True)
            nb += host_dw[k].numel() * host_dw[k].element_size()
        e1.record(up)
    torch.cuda.synchronize()
    up_gbs = nb / (e0.elapsed_time(e1) * 1e-3) / 1e9
    return {"value": n_elems * steps * world / secs, "unit": "elements/s",
            "h2d_bytes_per_step": h2d // steps, "d2h_bytes_per_step": d2h // steps,
            "ms_per_step": secs * 1e3 / steps, "repetitions_ms_per_step": [x * 1e3 / steps for x in rep_secs],
            "h2d_gbs_upload_alone": up_gbs,
            "overlap": "dW upload of the next step and message download of the previous step overlap "
                       "the computation; the message lengths come back before each decode"}


# ---------------------------------------------------------------- residue contrast
def run_residue_contrast(args):
    """The contrast of "AdaComp (Adaptive Residual Gradient Compression)", Claims >
    Mechanism #r629-self-adjusting-sparsity-prevents-residual-explosion, on synthetic
    gradients: one 4096x4096 layer, dW_t = 1e-3 (m + z_t) with a direction m ~ N(0, 0.25)
    kept for every step (gradients of a training run keep much of their direction)
    and fresh noise z_t ~ N(0, 1); the residue is carried for `contrast_steps` steps
    under AdaComp and under Local Selection (hard threshold, no soft-threshold probe)
    at L_T = 50, 500 and 5000. Reports, per step, the residue's min and max and the
    compression ratio (4N / message bytes), all through the C ABI."""
    import residual_gradient_compression_gb300 as ac
    from residual_gradient_compression_gb300 import build
    build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    n = 4096 * 4096
    g = torch.Generator(device=dev)
    g.manual_seed(5_000_000)
    m = torch.randn(n, generator=g, device=dev) * 0.5
    out = {"mode": "residue_contrast", "layer_elements": n, "steps": args.contrast_steps,
           "dW": "1e-3 * (m + z_t), m ~ N(0, 0.25) fixed, z_t ~ N(0, 1) fresh each step", "results": []}
    for L in (50, 500, 5000):
        for rule in (ac.RULE_ADACOMP, ac.RULE_LOCAL_SELECTION):
            h = ac.adacomp_init_layer(n, L, ac.F32)
            ac.adacomp_set_selection_rule(h, rule)
            msg = torch.zeros(h.max_msg_bytes[0], dtype=torch.uint8, device=dev)
            ws = torch.zeros(h.compress_ws_bytes, dtype=torch.uint8, device=dev)
            res = torch.zeros(n, device=dev)
            lo, hi, comp = [], [], []
            for t in range(args.contrast_steps):
                gz = torch.Generator(device=dev)
                gz.manual_seed(5_000_001 + t)
                dw = (m + torch.randn(n, generator=gz, device=dev)) * 1e-3
                ac.adacomp_compress(h, res, dw, msg, ws)
                mb, s, st = ac.adacomp_query(h, ws)
                if st != ac.OK:
                    raise RuntimeError(f"device status {st}")
                mn, mx = torch.aminmax(res)
                lo.append(float(mn))
                hi.append(float(mx))
                comp.append(4.0 * n / mb)
            out["results"].append({"bin_len": L, "rule": "adacomp" if rule == ac.RULE_ADACOMP else "local_selection",
                                   "residue_min": lo, "residue_max": hi, "compression": comp})
            ac.adacomp_free(h)
    return out


# ---------------------------------------------------------------- oracle legs
def oracle_sample_layers(args):
    """The layers one oracle step covers: the whole workload when it is small,
    otherwise a fixed slice of it (said in the JSON's `sample`)."""
    layers = workload_layers(args)
    if args.workload in ("resnet50", "fc400k"):
        return layers, "all layers"
    if args.workload == "flat100m":
        return layers, "one learner's 10^8-element layer per step (learners 0..15 in turn, each its own dW)"
    if args.workload == "lstm_fc":
        return [layers[0], layers[4]], "one LSTM tensor + one FC tensor (25.2M elements)"
    sub = [l for l in layers if l.name.startswith("h0.")]
    return sub, "all tensors of one decoder block (50.4M elements)"


def oracle_run(args, steps=None, budget_s=None, warmup=0):
    """Runs the oracle on host cores: compress of every sampled layer (one learner,
    carried residue) and decode of the step's messages. Returns (elements, seconds,
    steps, sample text); input generation is outside the timed part."""
    import oracle
    oracle.build()
    layers, sample = oracle_sample_layers(args)
    names = [l.name for l in workload_layers(args)]
    res = [np.zeros(l.numel, np.float32) for l in layers]
    dense = [np.zeros(l.numel, np.float32) for l in layers]
    elems = secs = 0.0
    done = 0
    i = 0
    K = learners(args)
    while True:
        dws = []
        for ly in layers:
            t = wl.gen_dw(args.workload, names.index(ly.name), ly, i // K, learner=i % K, device="cpu")
            dws.append(t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy())
        t0 = time.perf_counter()
        for ly, r, d, dn in zip(layers, res, dws, dense):
            out = oracle.compress(r, d, ly.bin_len)
            oracle.decode_accumulate(ly.numel, ly.bin_len, [out.msg], dn)
        dt = time.perf_counter() - t0
        i += 1
        if i <= warmup:
            continue
        secs += dt
        elems += sum(l.numel for l in layers)
        done += 1
        if steps is not None and done >= steps:
            break
        if budget_s is not None and secs >= budget_s:
            break
    what = (f"{args.workload}: {sample}, {done} step(s) of oracle compress + decode of that message, carried "
            "residue; inputs from the same seeded generators on the host")
    return elems, secs, done, what


def oracle_baseline(args):
    elems, secs, done, what = oracle_run(args, budget_s=args.cpu_seconds, steps=max(args.steps, 1))
    return {"value": elems / secs, "unit": "elements/s", "cores": 1, "kind": "oracle", "sample": what,
            "seconds": secs, "host": _host()}


def _host():
    try:
        model = ""
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
        return {"nproc": os.cpu_count(), "cpu": model, "arch": os.uname().machine}
    except Exception:
        return {"nproc": os.cpu_count()}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    elems, secs, done, what = oracle_run(args, steps=max(args.steps, 1), warmup=args.warmup)
    v = elems / secs
    layers = workload_layers(args)
    return {
        "metric": METRIC, "value": v, "unit": "elements/s", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": done, "warmup": args.warmup, "ms_per_step": secs * 1e3 / done, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16+f32" if layers[0].dw_dtype == "bf16" else "f32",
        "data": "synthetic", "impl": "reference",
        "config": bench_config(args, layers, learners(args), int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": {"value": v, "unit": "elements/s", "cores": 1, "kind": "oracle", "sample": what,
                         "host": _host()},
        "e2e": {"value": v, "unit": "elements/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    if args.impl == "reference":
        out = run_reference(args)
        if out is not None:
            print(json.dumps(out), flush=True)
        return 0
    rank, world = dist_init()
    if args.residue_contrast:
        if rank == 0:
            print(json.dumps(run_residue_contrast(args)), flush=True)
        return 0
    out, run = run_device(args, rank, world)
    del run
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = oracle_baseline(args)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
