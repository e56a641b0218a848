#!/usr/bin/env python3
"""Benchmark of the resharding engine and the 1D tensor-parallel MLP on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  * the resharding sweep on an activation tensor [B=8, S=2048, H=4096] in
    float32 and bf16, on virtual meshes 1x8 and 2x4, six transitions each
    (dims_mapping [0,-1,-1]->[-1,-1,0], [-1,-1,0]->[-1,0,-1],
    [0,-1,1]->[-1,-1,-1], P-sum of 8->B, P-sum of 8->S(2), B->S(0)): 24
    reshard calls, L2 flushed before each;
  * the tensor-parallel MLP X[8192,4096] . A[4096,16384] -> GELU ->
    . B[16384,4096], P = 8, bf16 in / float32 accumulate, fused reduction;
  * the Domino schedule on the Llama-70B MLP shape (tokens 4096, hidden 8192,
    ffn 28672, P = 8): row split into 2 chunks with the reduction of one chunk
    on a second stream, next to the serial (one stream) schedule.

`value` is the resharding throughput (algorithmic bytes of the 24 calls over
their device time); the MLP and Domino figures are reported beside it.
Inputs are seeded (torch's Philox generator on the device), resident in HBM
when the timed region starts. `--impl reference` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "reshard GB/s (% of HBM peak); TP-MLP TFLOP/s (% of bf16 peak), 1 GB300"
SWEEP_SHAPE = (8, 2048, 4096)
UNEVEN_SHAPE = (12289, 6143)
MLP = dict(M=8192, K=4096, F=16384, N=4096, P=8)
DOMINO = dict(M=4096, K=8192, F=28672, N=8192, P=8)
# The workload both arms report (the reference arm times a bounded sample of it).
CONFIG = {"workload": "resharding sweep [8,2048,4096] f32+bf16 on virtual meshes 1x8 and 2x4 (6 transitions each) "
                      "+ TP-MLP 8192x4096x16384x4096 P=8 + Domino 4096x8192x28672x8192 P=8",
          "parallelism": "virtual mesh of 8 ranks inside each GPU; GPUs run independent replicas",
          "l2": "flushed before every timed call: a 512 MiB write, then a 512 MiB read, so that no dirty line of "
                "the flush is written back inside the timed region"}
L2_FLUSH_BYTES = 512 * 1024 * 1024
# What the reference arm (the CPU oracle) times: a bounded sample of the
# resharding sweep, float32 only, on a slice of the activation tensor.
REFERENCE_CONFIG = {"workload": "resharding sweep sample: the 12 float32 transitions (meshes 1x8 and 2x4) on a "
                                "[8,256,4096] slice of the [8,2048,4096] activation tensor, called in turn",
                    "parallelism": "virtual mesh of 8 ranks, single-threaded CPU oracle on rank 0",
                    "l2": "host caches: each tensor is 32 MiB and the partials 256 MiB, larger than the host caches"}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), \
            "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ---- the sweep -----------------------------------------------------------------------

TRANSITIONS = [
    ("[0,-1,-1]->[-1,-1,0]", [0, -1, -1], [-1, -1, 0], False),
    ("[-1,-1,0]->[-1,0,-1]", [-1, -1, 0], [-1, 0, -1], False),
    ("[0,-1,1]->[-1,-1,-1]", [0, -1, 1], [-1, -1, -1], False),
    ("P8->B", None, [-1, -1, -1], True),
    ("P8->S(2)", None, [-1, -1, 0], True),
    ("B->S(0)", [-1, -1, -1], [0, -1, -1], False),
]


def sweep_specs(rtp, mesh_name):
    """(name, src spec, dst spec) of the six transitions on mesh '1x8' or '2x4'.
    On 1x8, mappings naming only mesh dim 0 use the 1-D mesh [8]; [0,-1,1]
    uses [1,8]. On 2x4, P-sum of 8 is partial over both mesh dims, and a
    destination split or a broadcast source over 'all 8' nests both mesh dims."""
    out = []
    for name, sdm, ddm, partial in TRANSITIONS:
        if mesh_name == "1x8":
            m = (1, 8) if (sdm and 1 in sdm) else (8,)
            if partial:
                src = rtp.spec_nd_sbp(m, ("P",))
            else:
                src = rtp.spec_from_dims_mapping(sdm, m)
            dst = rtp.spec_from_dims_mapping(ddm, m)
        else:
            m = (2, 4)
            full8 = partial or sdm == [-1, -1, -1]
            if partial:
                src = rtp.spec_nd_sbp(m, ("P", "P"))
            elif sdm == [-1, -1, -1]:
                src = rtp.spec_nd_sbp(m, ("B", "B"))
            else:
                src = rtp.spec_from_dims_mapping(sdm, m)
            ax = [i for i, v in enumerate(ddm) if v >= 0]
            if full8 and ax:
                dst = rtp.spec_nd_sbp(m, (("S", ax[0]), ("S", ax[0])))
            else:
                dst = rtp.spec_from_dims_mapping(ddm, m)
        out.append((name, src, dst, partial))
    return out


class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.file,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def _traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    source has not changed since the counters were taken (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    src = {"boxing_kernel": "boxing.cu", "tp_gemm_kernel": "tp_mlp.cu"}[kernel]
    with open(os.path.join(ROOT, "resharding_tensor_parallelism_gb300", "csrc", src), "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()[:16]
    with open(path) as f:
        for line in f:
            p = line.split()
            if len(p) >= 4 and not line.startswith("#") and p[0] == kernel and p[1] == workload and p[2] == digest:
                return float(p[3])
    return None


def reduce_over_ranks(dist, x: float, device, op: str = "max") -> float:
    """Max (or sum) of one float over the process group (x itself without one).
    Replicas report the slowest rank's time and the sum of their bytes."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def whole_job_gbs(bytes_per_rank: float, world: int, max_ms: float) -> float:
    """Whole-job throughput of N replicas: every rank moves bytes_per_rank;
    the job takes as long as the slowest rank."""
    return bytes_per_rank * world / (max_ms * 1e-3) / 1e9


def run_ours(args, rank, world, local_rank):
    import torch
    import resharding_tensor_parallelism_gb300 as rtp

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl", device_id=dev)
        dist = dist_mod
    rtp.lib()
    hbm_peak, bf16_peak, bf16_sust, peak_src = _peaks()
    gen = torch.Generator(device=dev)
    gen.manual_seed(1234 + 7919 * rank)

    def randn(shape, dtype, std=1.0):
        return (torch.randn(shape, generator=gen, device=dev, dtype=torch.float32) * std).to(dtype)

    # ---- sweep inputs: pieces resident in HBM ----
    # the flush buffers are at least 4x the L2 size the device reports
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0))
    flush_bytes = max(L2_FLUSH_BYTES, 4 * l2_bytes) // 4096 * 4096
    flush_w = torch.empty(flush_bytes // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones(flush_bytes // 4, dtype=torch.float32, device=dev)

    class _Flush:
        """L2 flush before a timed call: write a buffer larger than L2, then read
        another one, so that the write's dirty lines go back to HBM before the
        timed region instead of inside it (every call starts from a cold, clean L2)."""

        @staticmethod
        def zero_():
            flush_w.zero_()
            torch.sum(flush_r)

    flush = _Flush()
    sweep = []  # (label, dtype_code, src pieces, src, dst pieces, dst, bytes, launches)
    shards = []  # (label, full tensor, spec, pieces, bytes, launches): shard() of the sweep's S/B sources
    whole = rtp.spec_nd_sbp((1,), ("B",))
    for dtype, code in ((torch.float32, rtp.F32), (torch.bfloat16, rtp.BF16)):
        T = randn(SWEEP_SHAPE, dtype)
        partials = [randn(SWEEP_SHAPE, dtype) for _ in range(8)]
        for mesh_name in ("1x8", "2x4"):
            for name, src, dst, partial in sweep_specs(rtp, mesh_name):
                ins = partials if partial else rtp.shard(T, src)
                outs = [torch.empty(rtp.shard_shape(SWEEP_SHAPE, dst, r), dtype=dtype, device=dev)
                        for r in range(dst.num_ranks)]
                rd, wr, nt, nl = rtp.reshard_cost(code, SWEEP_SHAPE, src, dst)
                label = "%s %s %s" % (str(dtype).split(".")[-1], mesh_name, name)
                sweep.append((label, code, ins, src, outs, dst, rd + wr, nl))
                if not partial:
                    srd, swr, _, snl = rtp.reshard_cost(code, SWEEP_SHAPE, whole, src)
                    shards.append((label, T, src, ins, srd + swr, snl))
    # the uneven configuration: [12289, 6143] float32 U[-1,1) on a 2x2 mesh,
    # (S0,S1) -> (S1,S0) and (S0,S1) -> (B,S1)
    u_src = rtp.spec_nd_sbp((2, 2), (("S", 0), ("S", 1)))
    u_pieces = rtp.shard(torch.rand(UNEVEN_SHAPE, generator=gen, device=dev) * 2 - 1, u_src)
    uneven = []  # (label, src pieces, dst spec, dst pieces, bytes, launches)
    for name, ents in (("(S0,S1)->(S1,S0)", (("S", 1), ("S", 0))), ("(S0,S1)->(B,S1)", ("B", ("S", 1)))):
        dst = rtp.spec_nd_sbp((2, 2), ents)
        outs = [torch.empty(rtp.shard_shape(UNEVEN_SHAPE, dst, r), dtype=torch.float32, device=dev)
                for r in range(dst.num_ranks)]
        rd, wr, nt, nl = rtp.reshard_cost(rtp.F32, UNEVEN_SHAPE, u_src, dst)
        uneven.append((name, u_pieces, dst, outs, rd + wr, nl))
    torch.cuda.synchronize()

    # ---- MLP inputs ----
    def mlp_buffers(c, extra_partials):
        M, K, F, N, P = c["M"], c["K"], c["F"], c["N"], c["P"]
        X = randn((M, K), torch.bfloat16)
        A = [randn((K, F // P), torch.bfloat16, 0.02) for _ in range(P)]
        B = [randn((F // P, N), torch.bfloat16, 0.02) for _ in range(P)]
        Y = [torch.empty((M, F // P), dtype=torch.bfloat16, device=dev) for _ in range(P)]
        Z = torch.empty((M, N), dtype=torch.float32, device=dev)
        parts = [torch.empty((M, N), dtype=torch.float32, device=dev) for _ in range(P)] if extra_partials else None
        return dict(X=X, A=A, B=B, Y=Y, Z=Z, parts=parts, flops=2 * M * K * F + 2 * M * F * N)

    mlp = mlp_buffers(MLP, False)
    dom = mlp_buffers(DOMINO, True)
    # training: the forward that keeps H, and the backward from a bf16 dZ
    M_, K_, F_, N_, P_ = MLP["M"], MLP["K"], MLP["F"], MLP["N"], MLP["P"]
    trn = dict(H=[torch.empty((M_, F_ // P_), dtype=torch.bfloat16, device=dev) for _ in range(P_)],
               dZ=randn((M_, N_), torch.bfloat16),
               dH=[torch.empty((M_, F_ // P_), dtype=torch.bfloat16, device=dev) for _ in range(P_)],
               dX=torch.empty((M_, K_), dtype=torch.float32, device=dev),
               dA=[torch.empty((K_, F_ // P_), dtype=torch.float32, device=dev) for _ in range(P_)],
               dB=[torch.empty((F_ // P_, N_), dtype=torch.float32, device=dev) for _ in range(P_)],
               parts=[torch.empty((M_, K_), dtype=torch.float32, device=dev) for _ in range(P_)])
    # sequence parallel: X split by rows over the ranks, Z scattered by rows
    sp_rows = MLP["M"] // MLP["P"]
    sp_x = [mlp["X"][r * sp_rows:(r + 1) * sp_rows].contiguous() for r in range(MLP["P"])]
    sp_z = [torch.empty((sp_rows, MLP["N"]), dtype=torch.float32, device=dev) for _ in range(MLP["P"])]
    s1 = torch.cuda.Stream(device=dev)
    # the reduction alone: P-sum of the 8 float32 partials into one buffer
    dom_red_src = rtp.spec_nd_sbp((8,), ("P",))
    dom_red_dst = rtp.spec_nd_sbp((1,), ("B",))
    dom_shape = (DOMINO["M"], DOMINO["N"])

    def run_mlp():
        rtp.tp_mlp(mlp["X"], mlp["A"], mlp["B"], Y=mlp["Y"], Z=mlp["Z"], mode=1)

    def run_sp():
        rtp.tp_mlp_sp(sp_x, mlp["A"], mlp["B"], Y=mlp["Y"], Z_shards=sp_z)

    def domino(chunks, col_blocks, in_epilogue):
        """The Domino schedule: the rank partials summed in the row-parallel
        GEMM's epilogue (the default), or by kernels of their own on the
        second stream, after each window."""
        def run():
            prev = rtp.tp_mlp_overlap(1 if in_epilogue else 0)
            rtp.tp_mlp(dom["X"], dom["A"], dom["B"], Y=dom["Y"], partials=dom["parts"], Z=dom["Z"], mode=0,
                       chunks=chunks, col_blocks=col_blocks, s1=s1)
            rtp.tp_mlp_overlap(prev)
        return run

    def run_serial():
        """No overlap: the GEMMs, then one kernel sums the partials (one stream)."""
        prev = rtp.tp_mlp_overlap(0)
        rtp.tp_mlp(dom["X"], dom["A"], dom["B"], Y=dom["Y"], partials=dom["parts"], Z=dom["Z"], mode=0, chunks=1)
        rtp.tp_mlp_overlap(prev)

    def run_dom_fused():
        rtp.tp_mlp(dom["X"], dom["A"], dom["B"], Y=dom["Y"], Z=dom["Z"], mode=1)

    def run_reduce():
        rtp.reshard(dom["parts"], dom_shape, dom_red_src, dom_red_dst, out=[dom["Z"]])

    def run_train_fwd():
        rtp.tp_mlp_train_forward(mlp["X"], mlp["A"], mlp["B"], Y=mlp["Y"], H=trn["H"], Z=mlp["Z"])

    def run_bwd():
        rtp.tp_mlp_backward(mlp["X"], mlp["A"], mlp["B"], trn["H"], mlp["Y"], trn["dZ"], dH=trn["dH"], dX=trn["dX"],
                            dA=trn["dA"], dB=trn["dB"], mode=1)

    def bwd_overlap(in_epilogue):
        """Backward with the dX partials written and summed: in the dX GEMM's
        epilogue (the default) or by a kernel of its own on the second stream
        beside the weight-gradient GEMMs."""
        def run():
            prev = rtp.tp_mlp_overlap(1 if in_epilogue else 0)
            rtp.tp_mlp_backward(mlp["X"], mlp["A"], mlp["B"], trn["H"], mlp["Y"], trn["dZ"], dH=trn["dH"],
                                dX=trn["dX"], dA=trn["dA"], dB=trn["dB"], dX_partials=trn["parts"], mode=0, s1=s1)
            rtp.tp_mlp_overlap(prev)
        return run

    ops = [(label, (lambda c=c, i=i, s=s, o=o, d=d: rtp.reshard(i, SWEEP_SHAPE, s, d, out=o)), nbytes, nl)
           for (label, c, i, s, o, d, nbytes, nl) in sweep]
    shard_ops = [(label, (lambda T=T, sp=sp, o=o: rtp.shard(T, sp, out=o)), nbytes, nl)
                 for (label, T, sp, o, nbytes, nl) in shards]
    uneven_ops = [(label, (lambda i=i, d=d, o=o: rtp.reshard(i, UNEVEN_SHAPE, u_src, d, out=o)), nbytes, nl)
                  for (label, i, d, o, nbytes, nl) in uneven]
    # (kind, function, launches of the library's kernels per call)
    mlp_ops = [("mlp", run_mlp, 2), ("sp", run_sp, 2),
               # the pages' schedule: every window's sum a launch of its own on the second stream
               ("domino", domino(2, 1, False), 2 * 3), ("domino4", domino(4, 1, False), 4 * 3),
               ("domino2d", domino(2, 2, False), 2 * (1 + 2 * 2)),
               # the sums in the row-parallel GEMM's epilogue: the GEMM launches only
               ("domino_esum", domino(2, 1, True), 2 * 2), ("domino4_esum", domino(4, 1, True), 4 * 2),
               ("domino2d_esum", domino(2, 2, True), 2 * 3), ("domino1_esum", domino(1, 1, True), 2),
               ("serial", run_serial, 3), ("dom_fused", run_dom_fused, 2), ("reduce", run_reduce, 1),
               ("train_fwd", run_train_fwd, 2), ("bwd", run_bwd, 4),
               ("bwd_overlap", bwd_overlap(False), 5), ("bwd_overlap_esum", bwd_overlap(True), 4)]
    launches_per_step = (sum(x[3] for x in ops) + sum(x[3] for x in shard_ops) + sum(x[3] for x in uneven_ops) +
                         sum(x[2] for x in mlp_ops))
    E = lambda: torch.cuda.Event(enable_timing=True)

    def step(record):
        for label, fn, nbytes, nl in shard_ops:
            flush.zero_()
            e0, e1 = E(), E()
            e0.record()
            fn()
            e1.record()
            record.append(("shard", label, e0, e1, nbytes))
        for label, fn, nbytes, nl in ops:
            flush.zero_()
            e0, e1 = E(), E()
            e0.record()
            fn()
            e1.record()
            record.append(("reshard", label, e0, e1, nbytes))
        for label, fn, nbytes, nl in uneven_ops:
            flush.zero_()
            e0, e1 = E(), E()
            e0.record()
            fn()
            e1.record()
            record.append(("uneven", label, e0, e1, nbytes))
        for kind, fn, _ in mlp_ops:
            flush.zero_()
            e0, e1 = E(), E()
            e0.record()
            fn()
            e1.record()
            record.append((kind, kind, e0, e1, 0))

    for _ in range(args.warmup):
        step([])
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    records = []
    with ClockSampler(local_rank) as clocks:
        t0 = E()
        t1 = E()
        t0.record()
        for _ in range(args.steps):
            step(records)
        t1.record()
        torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    wall_ms = t0.elapsed_time(t1)
    per = {}
    for kind, label, e0, e1, nbytes in records:
        ms = e0.elapsed_time(e1)
        d = per.setdefault((kind, label), [0.0, 0, nbytes])
        d[0] += ms
        d[1] += 1
    reshard_ms = sum(v[0] for (k, _), v in per.items() if k == "reshard")
    reshard_bytes = sum(v[2] * v[1] for (k, _), v in per.items() if k == "reshard")
    mlp_ms = per[("mlp", "mlp")][0]
    avg = lambda kind: per[(kind, kind)][0] / args.steps
    ser_ms, dfu_ms, red_ms, sp_ms = avg("serial"), avg("dom_fused"), avg("reduce"), avg("sp")
    tf_ms, bwd_ms, bwo_ms, bwoe_ms = avg("train_fwd"), avg("bwd"), avg("bwd_overlap"), avg("bwd_overlap_esum")
    hide = lambda ms: round((ser_ms - ms) / red_ms, 3) if red_ms > 0 else None

    def max_over_ranks(x):
        return reduce_over_ranks(dist, x, dev, "max")

    def gbs_of(kind, pred=lambda label: True):
        ms = sum(v[0] for (k, l), v in per.items() if k == kind and pred(l))
        by = sum(v[2] * v[1] for (k, l), v in per.items() if k == kind and pred(l))
        return by / (ms * 1e-3) / 1e9 if ms > 0 else None

    red_bytes = 8 * DOMINO["M"] * DOMINO["N"] * 4 + DOMINO["M"] * DOMINO["N"] * 4
    # Domino schedules on the Llama-70B MLP shape (2 and 4 row chunks; 2 chunks x 2 column blocks of B)
    dom_rows = {}
    for kind, name in (("domino", "2_chunks"), ("domino4", "4_chunks"), ("domino2d", "2_chunks_2_column_blocks")):
        ms, ms_e = avg(kind), avg(kind + "_esum")
        dom_rows[name] = {"ms": round(ms, 4), "hiding": hide(ms), "ms_epilogue_sum": round(ms_e, 4),
                          "hiding_epilogue_sum": hide(ms_e)}
    ms1 = avg("domino1_esum")
    dom_rows["1_chunk_epilogue_sum"] = {"ms": round(ms1, 4), "hiding": hide(ms1)}
    host = host_inference_timings(rtp)
    rows = {
        "a1_shard": {"gbs": round(gbs_of("shard"), 1), "frac_hbm": round(gbs_of("shard") / hbm_peak, 4),
                     "calls_per_step": len(shard_ops)},
        "a2_reshard_S_B": {"gbs": round(gbs_of("reshard", lambda l: "P8" not in l), 1),
                           "frac_hbm": round(gbs_of("reshard", lambda l: "P8" not in l) / hbm_peak, 4)},
        "a3_reshard_P": {"gbs": round(gbs_of("reshard", lambda l: "P8" in l), 1),
                         "frac_hbm": round(gbs_of("reshard", lambda l: "P8" in l) / hbm_peak, 4)},
        "a2_uneven_2x2": {"gbs": round(gbs_of("uneven"), 1), "frac_hbm": round(gbs_of("uneven") / hbm_peak, 4),
                          "per_call_gbs": {label: round(v[2] * v[1] / (v[0] * 1e-3) / 1e9, 1)
                                           for (k, label), v in per.items() if k == "uneven"},
                          "shape": "[12289,6143] float32 on 2x2 from (S0,S1)"},
        "a4_infer_spmd": {"us_per_call": host["infer_spmd_us"], "where": "host"},
        "a4p_reshape_rule": {"us_per_call": host["infer_reshape_us"], "where": "host"},
        "a7_reduce_separate": {"ms": round(red_ms, 4), "gbs": round(red_bytes / (red_ms * 1e-3) / 1e9, 1),
                               "frac_hbm": round(red_bytes / (red_ms * 1e-3) / 1e9 / hbm_peak, 4),
                               "shape": "8 float32 partials [4096,8192] -> Z"},
        "a6_a7_separate_schedule": {"ms": round(ser_ms, 4), "tflops": round(DOMINO_FLOPS / (ser_ms * 1e-3) / 1e12, 1)},
        "a5_a7_fused_domino_shape": {"ms": round(dfu_ms, 4), "tflops": round(DOMINO_FLOPS / (dfu_ms * 1e-3) / 1e12, 1),
                                     "frac_bf16": round(DOMINO_FLOPS / (dfu_ms * 1e-3) / 1e12 / bf16_peak, 4)},
        "f2_tp_mlp_sequence_parallel": {"ms": round(sp_ms, 4), "tflops": round(MLP_FLOPS / (sp_ms * 1e-3) / 1e12, 1),
                                        "frac_bf16": round(MLP_FLOPS / (sp_ms * 1e-3) / 1e12 / bf16_peak, 4)},
        "f3_infer_sbp_signature": {"us_per_call": host["sbp_signature_us"], "where": "host"},
        "f3_onnx_broadcast_checker": {"us_per_call": host["infer_broadcast_us"], "where": "host"},
        "a2_small_reshard_latency": small_reshard_latency(rtp, torch, dev),
        "cfg_tiny_latency": tiny_configuration_latency(rtp, torch, dev),
        "f1_tp_mlp_backward": {"ms": round(bwd_ms, 4), "tflops": round(2 * MLP_FLOPS / (bwd_ms * 1e-3) / 1e12, 1),
                               "frac_bf16": round(2 * MLP_FLOPS / (bwd_ms * 1e-3) / 1e12 / bf16_peak, 4),
                               "dX_sum": "fused in the GEMM",
                               "ms_separate_dX_sum_second_stream": round(bwo_ms, 4),
                               "ms_separate_dX_sum_in_epilogue": round(bwoe_ms, 4),
                               "train_forward_ms": round(tf_ms, 4),
                               "train_forward_tflops": round(MLP_FLOPS / (tf_ms * 1e-3) / 1e12, 1),
                               "traffic": _traffic("tp_gemm_kernel", "mlp_backward")},
    }
    reshard_ms = max_over_ranks(reshard_ms)
    mlp_ms = max_over_ranks(mlp_ms)
    wall_ms = max_over_ranks(wall_ms)
    gbs = whole_job_gbs(reshard_bytes, world, reshard_ms)
    tflops = MLP_FLOPS * args.steps * world / (mlp_ms * 1e-3) / 1e12
    per_launch_gbs = reshard_bytes / (reshard_ms * 1e-3) / 1e9
    tp_frac = round(tflops / world / bf16_peak, 4)
    rows["a5_a6_a7_tp_mlp_fused"] = {"tflops": round(tflops / world, 1), "frac_bf16": tp_frac}
    # The order of the keys puts both halves of the metric (resharding GB/s,
    # TP-MLP TFLOP/s) and the Domino figures at the end of the line.
    result = {
        "metric": METRIC,
        "value": round(gbs, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(wall_ms / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32+bf16",
        "data": "synthetic (seeded Philox normals on the device)",
        "config": dict(CONFIG, l2_cache_bytes=l2_bytes, l2_flush_bytes=flush_bytes),
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
        "rows": rows,
        "per_transition_gbs": {label: round(v[2] * v[1] / (v[0] * 1e-3) / 1e9, 1)
                               for (k, label), v in per.items() if k == "reshard"},
        "psum_error": psum_errors(rtp, torch, sweep),
        "roofline": {"bound": "hbm", "kernel": "boxing_kernel", "achieved": round(per_launch_gbs, 1),
                     "peak": hbm_peak, "unit": "GB/s", "frac": round(per_launch_gbs / hbm_peak, 4),
                     "peak_source": peak_src, "traffic": _traffic("boxing_kernel", "sweep")},
    }
    if rank == 0 and not args.no_e2e:
        result["e2e"] = e2e_sweep(rtp, torch, dev, sweep)
    lib_cmp = library_gemm_same_run(torch, mlp, run_mlp, flush) if rank == 0 and not args.no_library_gemm else None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(max_seconds=args.cpu_seconds, with_mlp=True)
    # The MLP is timed inside a long step (seconds of back-to-back work at the
    # power cap), so its roofline is the sustained bf16 figure; the burst
    # figure's fraction is given beside it.
    result["tp_mlp"] = {"value": round(tflops, 1), "unit": "TFLOP/s", "mode": "fused reduction",
                        "shape": "8192x4096x16384x4096 P=8", "ms_per_call": round(mlp_ms / args.steps, 4),
                        "roofline": {"bound": "tensor", "kernel": "tp_gemm_kernel", "achieved": round(tflops / world, 1),
                                     "peak": bf16_sust, "peak_kind": "sustained (timed inside a long step)",
                                     "unit": "TFLOP/s", "frac": round(tflops / world / bf16_sust, 4),
                                     "frac_of_burst": tp_frac, "burst_peak": bf16_peak,
                                     "peak_source": peak_src, "traffic": _traffic("tp_gemm_kernel", "mlp")},
                        "backward_tflops": rows["f1_tp_mlp_backward"]["tflops"],
                        "backward_frac": rows["f1_tp_mlp_backward"]["frac_bf16"]}
    if lib_cmp is not None:
        result["tp_mlp"]["beside_library_gemm"] = lib_cmp
    result["domino"] = {"shape": "4096x8192x28672x8192 P=8", "ms_serial": round(ser_ms, 4),
                        "ms_reduce_alone": round(red_ms, 4), "ms_fused": round(dfu_ms, 4), **dom_rows,
                        "tflops_2_chunks": round(DOMINO_FLOPS / (avg("domino") * 1e-3) / 1e12, 1)}
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def library_gemm_same_run(torch, mlp, run_mlp, flush, reps: int = 7):
    """The fused TP-MLP beside the library GEMM (torch.mm, i.e. cuBLAS) on the
    same problem, in the same process and at the same clocks: Y = X [A_0..A_7]
    and Z = Y [B_0; ..; B_7] as two plain bf16 GEMMs (8192x16384x4096 and
    8192x4096x16384), alternated with the library's own call, L2 flushed
    before each. For comparison only: the library GEMMs compute no GELU and
    write Z in bf16 (ours float32), so they do slightly less work. Medians."""
    X, A, B = mlp["X"], mlp["A"], mlp["B"]
    a_cat = torch.cat(A, dim=1)
    b_cat = torch.cat(B, dim=0)
    y_cat = torch.empty((X.shape[0], a_cat.shape[1]), dtype=torch.bfloat16, device=X.device)
    z_lib = torch.empty((X.shape[0], b_cat.shape[1]), dtype=torch.bfloat16, device=X.device)

    def lib():
        torch.mm(X, a_cat, out=y_cat)
        torch.mm(y_cat, b_cat, out=z_lib)

    def one(fn):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        return e0, e1

    for _ in range(3):
        one(lib)
        one(run_mlp)
    ours, theirs = [], []
    for _ in range(reps):
        theirs.append(one(lib))
        ours.append(one(run_mlp))
    torch.cuda.synchronize()
    med = lambda ev: statistics.median(a.elapsed_time(b) for a, b in ev)
    ms_ours, ms_lib = med(ours), med(theirs)
    del a_cat, b_cat, y_cat, z_lib
    return {"ms": round(ms_ours, 4), "tflops": round(MLP_FLOPS / (ms_ours * 1e-3) / 1e12, 1),
            "library_ms": round(ms_lib, 4), "library_tflops": round(MLP_FLOPS / (ms_lib * 1e-3) / 1e12, 1),
            "speedup_over_library": round(ms_lib / ms_ours, 4),
            "library": "torch.mm (cuBLAS) bf16: X[A_i] then Y[B_i], bf16 outputs, no GELU; alternated with ours, "
                       "L2 flushed before each, median of %d" % reps}


def psum_errors(rtp, torch, sweep):
    """Error of the float32 partial sums of the sweep (P-sum of 8 -> B and ->
    S(2), meshes 1x8 and 2x4) against their exact sums, taken in float64 on
    the device from the same partials: the normwise max|err| / max|exact| and
    the element-wise max |err| / sum_i |x_i| (the condition-aware form; both
    bounded by 1e-6). Every destination piece is compared."""
    out = {}
    for label, code, ins, src, outs, dst, _, _ in sweep:
        if code != rtp.F32 or "P8" not in label:
            continue
        exact = torch.zeros(ins[0].shape, dtype=torch.float64, device=ins[0].device)
        mag = torch.zeros_like(exact)
        for x in ins:
            exact += x.double()
            mag += x.double().abs()
        err = torch.zeros_like(exact)
        covered = torch.zeros(exact.shape, dtype=torch.bool, device=exact.device)
        for r in range(dst.num_ranks):
            lo, hi, _ = rtp.shard_box(SWEEP_SHAPE, dst, r)
            sl = tuple(slice(a, b) for a, b in zip(lo, hi))
            e = (outs[r].double() - exact[sl]).abs()
            err[sl] = torch.maximum(err[sl], e)
            covered[sl] = True
        assert bool(covered.all())
        out[label] = {"normwise": float(err.max() / exact.abs().max()),
                      "elementwise_over_sum_abs": float((err / mag.clamp_min(1e-300)).max())}
        del exact, mag, err, covered
    torch.cuda.empty_cache()
    return out


def tiny_cases(torch, dev):
    """The tiny exactness configuration on the device: the [[1,2],[3,4]] ONNX
    splits, broadcast and split+broadcast, the OneFlow S(1) -> S(0) reshard of
    the add example's second input, a P-sum of 4 [4,6] partials to B, and the
    [4,8] x [8,16] x [16,8] MLP on 2 ranks (bf16)."""
    import resharding_tensor_parallelism_gb300 as rtp

    g = torch.Generator(device=dev)
    g.manual_seed(0)
    T = torch.tensor([[1.0, 2.0], [3.0, 4.0]], device=dev)
    T8 = torch.arange(1, 9, dtype=torch.float32, device=dev).view(2, 4)
    onnx = {"split axes 0 and 1 on 4 devices": ([0, 1, 2, 3], {}, [(0, 2), (1, 2)]),
            "broadcast through device_map": ([-1], {-1: [0, 1]}, []),
            "split axis 0, each piece broadcast to its group": ([-1, -2], {-1: [0, 1], -2: [2, 3]}, [(0, 2)])}
    ops = {}
    for name, (device, dmap, sd) in onnx.items():
        spec = rtp.spec_from_onnx(2, device, dmap, sd)
        out = rtp.shard(T, spec)
        ops["shard: " + name] = lambda spec=spec, out=out: rtp.shard(T, spec, out=out)
    s0, s1 = rtp.spec_nd_sbp((2,), (("S", 0),)), rtp.spec_nd_sbp((2,), (("S", 1),))
    t2 = rtp.shard(T8, s1)
    t2o = rtp.reshard(t2, (2, 4), s1, s0)
    ops["reshard S(1) -> S(0), [2,4] on 2 ranks"] = lambda: rtp.reshard(t2, (2, 4), s1, s0, out=t2o)
    parts = [torch.randn((4, 6), generator=g, device=dev) for _ in range(4)]
    sp, sb = rtp.spec_nd_sbp((4,), ("P",)), rtp.spec_nd_sbp((4,), ("B",))
    pb = rtp.reshard(parts, (4, 6), sp, sb)
    ops["reshard P -> B, 4 partials [4,6]"] = lambda: rtp.reshard(parts, (4, 6), sp, sb, out=pb)
    X = torch.randn((4, 8), generator=g, device=dev).bfloat16()
    A = [torch.randn((8, 8), generator=g, device=dev).bfloat16() for _ in range(2)]
    B = [torch.randn((8, 8), generator=g, device=dev).bfloat16() for _ in range(2)]
    Z, Y = rtp.tp_mlp(X, A, B)
    ops["tp_mlp [4,8] x [8,16] x [16,8], P=2"] = lambda: rtp.tp_mlp(X, A, B, Y=Y, Z=Z, mode=1)
    return ops


def tiny_configuration_latency(rtp, torch, dev, n: int = 100):
    """Latency of each call of the tiny configuration, issued back to back as
    direct calls (host checks, planning and launch every call): microseconds
    per call from CUDA events. Latency-bound, so no roofline applies."""
    out = {}
    E = lambda: torch.cuda.Event(enable_timing=True)
    for name, fn in tiny_cases(torch, dev).items():
        for _ in range(10):
            fn()
        torch.cuda.synchronize()
        e0, e1 = E(), E()
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        out[name] = round(e0.elapsed_time(e1) * 1e3 / n, 2)
    return {"us_per_call": out, "calls_each": n}


def cpu_tiny_baseline(n: int = 200):
    """The oracle on the tiny configuration, the same operations as
    tiny_cases: microseconds per call, one core."""
    import numpy as np

    import oracle
    import synth

    T = np.array([[1, 2], [3, 4]], np.float32)
    T8 = np.arange(1, 9, dtype=np.float32).reshape(2, 4)
    onnx = {"split axes 0 and 1 on 4 devices": ([0, 1, 2, 3], {}, [(0, 2), (1, 2)]),
            "broadcast through device_map": ([-1], {-1: [0, 1]}, []),
            "split axis 0, each piece broadcast to its group": ([-1, -2], {-1: [0, 1], -2: [2, 3]}, [(0, 2)])}
    ops = {}
    for name, (device, dmap, sd) in onnx.items():
        lay = oracle.layout_from_onnx(2, device, dmap, sd)
        ops["shard: " + name] = lambda lay=lay: oracle.shard(T, lay)
    L0, L1 = oracle.Layout((2,), (("S", 0),)), oracle.Layout((2,), (("S", 1),))
    t2 = oracle.shard(T8, L1)
    ops["reshard S(1) -> S(0), [2,4] on 2 ranks"] = lambda: oracle.reshard(t2, (2, 4), L1, L0)
    parts = [synth.normal(100 + k, (4, 6), "f32") for k in range(4)]
    LP, LB = oracle.Layout((4,), ("P",)), oracle.Layout((4,), ("B",))
    ops["reshard P -> B, 4 partials [4,6]"] = lambda: oracle.reshard(parts, (4, 6), LP, LB)
    X = synth.normal(0, (4, 8), "bf16")
    A = [synth.normal(1 + i, (8, 8), "bf16") for i in range(2)]
    B = [synth.normal(3 + i, (8, 8), "bf16") for i in range(2)]
    ops["tp_mlp [4,8] x [8,16] x [16,8], P=2"] = lambda: oracle.tp_mlp(X, A, B)
    out = {}
    for name, fn in ops.items():
        fn()
        t = time.perf_counter()
        for _ in range(n):
            fn()
        out[name] = round((time.perf_counter() - t) / n * 1e6, 2)
    return {"us_per_call": out, "cores": 1, "kind": "oracle", "calls_each": n}


def small_reshard_latency(rtp, torch, dev, n: int = 100):
    """Latency of a small reshard (a [8,64,512] float32 activation, S(0) -> S(2)
    on the 1x8 mesh, 1 MiB) issued back to back: direct calls (host planning
    and launch on every call) against the same calls replayed from a CUDA
    graph; microseconds per call."""
    shape = (8, 64, 512)
    s0, s2 = rtp.spec_nd_sbp((8,), (("S", 0),)), rtp.spec_nd_sbp((8,), (("S", 2),))
    src = rtp.shard(torch.randn(shape, device=dev), s0)
    out = [torch.empty(rtp.shard_shape(shape, s2, r), device=dev) for r in range(8)]
    stream = torch.cuda.Stream(device=dev)
    E = lambda: torch.cuda.Event(enable_timing=True)

    def calls():
        for _ in range(n):
            rtp.reshard(src, shape, s0, s2, out=out, stream=stream)

    with torch.cuda.stream(stream):
        calls()
    torch.cuda.synchronize()
    e0, e1 = E(), E()
    e0.record(stream)
    calls()
    e1.record(stream)
    torch.cuda.synchronize()
    direct = e0.elapsed_time(e1) * 1e3 / n
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        calls()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = E(), E()
    e0.record(stream)
    with torch.cuda.stream(stream):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    replay = e0.elapsed_time(e1) * 1e3 / n
    return {"us_per_call_direct": round(direct, 2), "us_per_call_graph": round(replay, 2),
            "shape": "[8,64,512] f32, S(0)->S(2) on 1x8, calls back to back"}


def host_inference_timings(rtp, reps: int = 2000):
    """Host-side inference: the Paddle matmul example (mk,kn->mn on a 2D mesh)
    and the reshape [2,3,4096] -> [6,4096]; microseconds per call."""
    t = time.perf_counter()
    for _ in range(reps):
        rtp.infer_spmd("mk,kn->mn", [[0, -1], [-1, 1]], 2)
    a = (time.perf_counter() - t) / reps * 1e6
    t = time.perf_counter()
    for _ in range(reps):
        rtp.infer_reshape([2, 3, 4096], [0, -1, -1], [6, 4096], [2])
    b = (time.perf_counter() - t) / reps * 1e6
    t = time.perf_counter()
    for _ in range(reps):
        rtp.infer_sbp_signature((2, 4), 4, [[("S", 0)], [("S", 1)]])
    c = (time.perf_counter() - t) / reps * 1e6
    # ONNX broadcast rule: Add([4096,1],[1,4096]) with the page's composition layouts
    sa = rtp.spec_nd_sbp((2, 2), (("S", 0), "B"), (0, 1, 2, 3))
    sb = rtp.spec_nd_sbp((2, 2), (("S", 1), "B"), (0, 2, 1, 3))
    t = time.perf_counter()
    for _ in range(reps):
        rtp.infer_broadcast([(4096, 1), (1, 4096)], [sa, sb])
    d = (time.perf_counter() - t) / reps * 1e6
    return {"infer_spmd_us": round(a, 2), "infer_reshape_us": round(b, 2), "sbp_signature_us": round(c, 2),
            "infer_broadcast_us": round(d, 2)}


MLP_FLOPS = 2 * MLP["M"] * MLP["K"] * MLP["F"] + 2 * MLP["M"] * MLP["F"] * MLP["N"]
DOMINO_FLOPS = 2 * DOMINO["M"] * DOMINO["K"] * DOMINO["F"] + 2 * DOMINO["M"] * DOMINO["F"] * DOMINO["N"]


def e2e_sweep(rtp, torch, dev, sweep):
    """The sweep's bf16 1x8 transitions through the public API with host
    buffers: pinned host -> device copy of the source pieces, reshard, device
    -> pinned host copy of the destination pieces, all inside the timed region
    (2 timed steps after 1 warm-up). The six transitions of a step are
    pipelined on three streams, as a caller would, in the order that keeps both
    copy directions busy: the host-to-device copy of
    transition i+1 and the device-to-host copy of transition i-1 run while
    transition i reshards (the two copy directions use separate copy engines).
    Device buffers are allocated once, outside the timed region."""
    sel = [s for s in sweep if s[0].startswith("bfloat16 1x8")]
    # Order for a two-stage pipeline (upload, then download; the reshard in
    # between is short) by Johnson's rule: transitions that upload less than
    # they download first, by increasing upload; then the rest by decreasing
    # download. Both copy directions then stay busy from start to end.
    nb = lambda ps: sum(p.numel() * p.element_size() for p in ps)
    up = [x for x in sel if nb(x[2]) < nb(x[4])]
    rest = [x for x in sel if nb(x[2]) >= nb(x[4])]
    sel = sorted(up, key=lambda x: nb(x[2])) + sorted(rest, key=lambda x: -nb(x[4]))
    host_in = [[torch.empty(p.shape, dtype=p.dtype, pin_memory=True).copy_(p) for p in s[2]] for s in sel]
    host_out = [[torch.empty(p.shape, dtype=p.dtype, pin_memory=True) for p in s[4]] for s in sel]
    dev_in = [[torch.empty_like(p, device=dev) for p in hs] for hs in host_in]
    dev_out = [[torch.empty_like(p, device=dev) for p in hs] for hs in host_out]
    h2d = sum(p.numel() * p.element_size() for hs in host_in for p in hs)
    d2h = sum(p.numel() * p.element_size() for hs in host_out for p in hs)
    nbytes = sum(s[6] for s in sel)
    s_in, s_cmp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))

    def one():
        for i, s in enumerate(sel):
            with torch.cuda.stream(s_in):
                for d, h in zip(dev_in[i], host_in[i]):
                    d.copy_(h, non_blocking=True)
            e_in = torch.cuda.Event()
            e_in.record(s_in)
            s_cmp.wait_event(e_in)
            rtp.reshard(dev_in[i], SWEEP_SHAPE, s[3], s[5], out=dev_out[i], stream=s_cmp)
            e_c = torch.cuda.Event()
            e_c.record(s_cmp)
            s_out.wait_event(e_c)
            with torch.cuda.stream(s_out):
                for h, d in zip(host_out[i], dev_out[i]):
                    h.copy_(d, non_blocking=True)
        torch.cuda.synchronize()

    def uploads():
        with torch.cuda.stream(s_in):
            for i in range(len(sel)):
                for d, h in zip(dev_in[i], host_in[i]):
                    d.copy_(h, non_blocking=True)

    def downloads():
        with torch.cuda.stream(s_out):
            for i in range(len(sel)):
                for h, d in zip(host_out[i], dev_out[i]):
                    h.copy_(d, non_blocking=True)

    def timed(fn, reps=2):
        fn()
        torch.cuda.synchronize()
        t = time.perf_counter()
        for _ in range(reps):
            fn()
            torch.cuda.synchronize()
        return (time.perf_counter() - t) / reps

    one()
    t = time.perf_counter()
    for _ in range(2):
        one()
    dt = (time.perf_counter() - t) / 2
    # What the host link allows for this workload: each direction's copies
    # alone (same streams, no reshard); with the two directions fully
    # overlapped the copies take at least as long as the slower one. Both
    # directions started at once are reported too: they sometimes run far
    # below either direction alone.
    t_up, t_down = timed(uploads), timed(downloads)
    t_both = timed(lambda: (uploads(), downloads()))
    dt_link = max(t_up, t_down)
    return {"value": round(nbytes / dt / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "h2d_d2h_gbs": round((h2d + d2h) / dt / 1e9, 1),
            "link_ceiling_gbs": round(nbytes / dt_link / 1e9, 1),
            "frac_of_link_ceiling": round(dt_link / dt, 4),
            "link_h2d_gbs": round(h2d / t_up / 1e9, 1), "link_d2h_gbs": round(d2h / t_down / 1e9, 1),
            "link_both_at_once_gbs": round((h2d + d2h) / t_both / 1e9, 1),
            "frac_of_both_at_once": round(t_both / dt, 4),
            "workload": "the six bf16 transitions on the 1x8 mesh, host pinned buffers in and out, pipelined on "
                        "three streams; link_ceiling_gbs: the same copies with both directions fully overlapped "
                        "(the slower direction's copies alone); frac_of_both_at_once: the same copies, both "
                        "directions started together, no reshard, against the e2e step"}


# ---- CPU oracle (baseline and reference arm) ---------------------------------------------

CPU_SAMPLE_SHAPE = (8, 256, 4096)


def cpu_sample_cases():
    """The bounded sample the oracle runs: the twelve float32 transitions of
    the sweep (meshes 1x8 and 2x4) on a [8,256,4096] slice of the activation
    tensor (32 MiB per tensor, 256 MiB of partials, so it does not sit in the
    host caches). Returns (label, pieces, src, dst, distinct source bytes)."""
    import oracle
    import synth

    shape = CPU_SAMPLE_SHAPE
    T = synth.normal(11, shape, "f32")
    parts = [synth.normal(20 + k, shape, "f32") for k in range(8)]
    cases = []
    for mesh_name in ("1x8", "2x4"):
        for name, sdm, ddm, partial in TRANSITIONS:
            src, dst = _oracle_specs(oracle, mesh_name, sdm, ddm, partial)
            pieces = parts if partial else oracle.shard(T, src)
            nbytes = sum(p.nbytes for p in _distinct_reads(pieces, src, oracle, shape))
            cases.append((mesh_name + " " + name, pieces, src, dst, nbytes))
    return cases


def cpu_baseline(max_seconds: float = 12.0, with_mlp: bool = False, cases=None):
    """The oracle (single-threaded C++) on the bounded sample of
    `cpu_sample_cases`, call after call through the twelve transitions until
    about `max_seconds` of oracle time (at least one whole pass). GB/s of
    algorithmic bytes: distinct source bytes read plus destination bytes
    written."""
    import oracle

    if cases is None:
        cases = cpu_sample_cases()
    shape = CPU_SAMPLE_SHAPE
    total_bytes, total_s, done = 0, 0.0, 0
    while done < len(cases) or total_s < max_seconds:
        label, pieces, src, dst, nread = cases[done % len(cases)]
        t = time.perf_counter()
        outs = oracle.reshard(pieces, shape, src, dst)
        total_s += time.perf_counter() - t
        total_bytes += nread + sum(o.nbytes for o in outs)
        done += 1
    out = {"value": round(total_bytes / total_s / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": "%d float32 reshard calls (the sweep's 12 transitions, meshes 1x8 and 2x4, in turn) on a "
                     "[%d,%d,%d] slice of the activation tensor" % ((done,) + tuple(shape)),
           "seconds": round(total_s, 2), "host_cores": os.cpu_count()}
    if with_mlp:
        out["tp_mlp"] = cpu_mlp_baseline()
        out["tiny"] = cpu_tiny_baseline()
    return out


def cpu_mlp_baseline(rows: int = 64):
    """The oracle's TP-MLP (float64) on `rows` rows of the 8192x4096x16384x4096
    configuration, all columns; TFLOP/s of the sample (its full-size time is
    the sample time x 8192 / rows)."""
    import numpy as np

    import oracle
    import synth

    M, K, F, N, P = MLP["M"], MLP["K"], MLP["F"], MLP["N"], MLP["P"]
    X = synth.normal(40, (rows, K), "bf16")
    A = synth.normal(41, (K, F), "bf16", std=0.02)
    B = synth.normal(42, (F, N), "bf16", std=0.02)
    As = [np.ascontiguousarray(a) for a in np.split(A, P, axis=1)]
    Bs = [np.ascontiguousarray(b) for b in np.split(B, P, axis=0)]
    t = time.perf_counter()
    oracle.tp_mlp(X, As, Bs)
    dt = time.perf_counter() - t
    flops = 2 * rows * K * F + 2 * rows * F * N
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": "%d rows of Z (all 4096 columns) of the 8192x4096x16384x4096 P=8 MLP" % rows,
            "seconds": round(dt, 2), "full_size_seconds_extrapolated": round(dt * M / rows, 1)}


def _distinct_reads(pieces, layout, oracle, shape):
    """Source pieces counted once per distinct piece (broadcast replicas read once)."""
    seen, out = set(), []
    for r, p in enumerate(pieces):
        lo, hi, hv = oracle.shard_box(shape, layout, r)
        key = (lo, hi) if "P" not in layout.entries else r
        if key in seen or p.size == 0:
            continue
        seen.add(key)
        out.append(p)
    return out


def _oracle_specs(oracle, mesh_name, sdm, ddm, partial):
    if mesh_name == "1x8":
        m = (1, 8) if (sdm and 1 in sdm) else (8,)
        src = oracle.Layout(m, ("P",)) if partial else oracle.layout_from_dims_mapping(sdm, m)
        dst = oracle.layout_from_dims_mapping(ddm, m)
        return src, dst
    m = (2, 4)
    full8 = partial or sdm == [-1, -1, -1]
    if partial:
        src = oracle.Layout(m, ("P", "P"))
    elif sdm == [-1, -1, -1]:
        src = oracle.Layout(m, ("B", "B"))
    else:
        src = oracle.layout_from_dims_mapping(sdm, m)
    ax = [i for i, v in enumerate(ddm) if v >= 0]
    dst = oracle.Layout(m, (("S", ax[0]), ("S", ax[0]))) if (full8 and ax) else oracle.layout_from_dims_mapping(ddm, m)
    return src, dst


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle as it stands, on the host cores, rank 0 only."""
    if rank != 0:
        return
    per_step = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    cases = cpu_sample_cases()
    for _ in range(args.warmup):
        cpu_baseline(max_seconds=per_step, cases=cases)
    t = time.perf_counter()
    vals = [cpu_baseline(max_seconds=per_step, cases=cases) for _ in range(args.steps)]
    wall = time.perf_counter() - t
    v = statistics.median(x["value"] for x in vals)
    cb = dict(vals[-1])
    cb["value"] = v
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(wall / args.steps * 1e3, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded generator)",
        "config": dict(REFERENCE_CONFIG),
        "cpu_baseline": cb, "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


PROFILE_CASES = {
    # name: (kind, details)
    "reshard_f32_s0s2": ("reshard", ("1x8", 0, "f32")),
    "reshard_bf16_s0s2": ("reshard", ("1x8", 0, "bf16")),
    "reshard_f32_p8b": ("reshard", ("1x8", 3, "f32")),
    "reshard_f32_p8s2": ("reshard", ("1x8", 4, "f32")),
    "reshard_f32_s0s2b": ("reshard", ("1x8", 2, "f32")),
    "reshard_bf16_s2s1": ("reshard", ("1x8", 1, "bf16")),
    "sweep": ("sweep", None),
    "mlp_fused": ("mlp", MLP),
    "domino_fused": ("mlp", DOMINO),
    "mlp_backward": ("mlp_backward", MLP),
    "mlp_beside_library": ("mlp_library", MLP),
    "uneven": ("uneven", None),
}


def run_profile_case(name: str, repeats: int = 2):
    """A small, fixed workload for an ncu capture: `repeats` calls of one
    operation on inputs generated on the device (no other library launches)."""
    import torch
    import resharding_tensor_parallelism_gb300 as rtp

    torch.cuda.set_device(0)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    kind, det = PROFILE_CASES[name]
    if kind == "sweep":
        # the 24 reshard calls of one bench step, in bench order, one launch each
        order = []
        for dtype, code in ((torch.float32, rtp.F32), (torch.bfloat16, rtp.BF16)):
            for mesh_name in ("1x8", "2x4"):
                for tname, src, dst, partial in sweep_specs(rtp, mesh_name):
                    ins = [torch.randn(rtp.shard_shape(SWEEP_SHAPE, src, r), generator=gen, device="cuda").to(dtype)
                           for r in range(src.num_ranks)]
                    outs = [torch.empty(rtp.shard_shape(SWEEP_SHAPE, dst, r), dtype=dtype, device="cuda")
                            for r in range(dst.num_ranks)]
                    rd, wr, nt, nl = rtp.reshard_cost(code, SWEEP_SHAPE, src, dst)
                    torch.cuda.synchronize()
                    rtp.reshard(ins, SWEEP_SHAPE, src, dst, out=outs)
                    torch.cuda.synchronize()
                    order.append({"call": "%s %s %s" % (str(dtype).split(".")[-1], mesh_name, tname),
                                  "algorithmic_bytes": rd + wr, "launches": nl})
                    del ins, outs
                    torch.cuda.empty_cache()
        print(json.dumps({"case": name, "calls": order}))
    elif kind == "uneven":
        # [12289, 6143] float32 on 2x2: (S0,S1) -> (S1,S0), then (S0,S1) -> (B,S1), one launch each
        src = rtp.spec_nd_sbp((2, 2), (("S", 0), ("S", 1)))
        ins = rtp.shard(torch.rand(UNEVEN_SHAPE, generator=gen, device="cuda") * 2 - 1, src)
        order = []
        for tname, ents in (("(S0,S1)->(S1,S0)", (("S", 1), ("S", 0))), ("(S0,S1)->(B,S1)", ("B", ("S", 1)))):
            dst = rtp.spec_nd_sbp((2, 2), ents)
            outs = [torch.empty(rtp.shard_shape(UNEVEN_SHAPE, dst, r), device="cuda") for r in range(dst.num_ranks)]
            rd, wr, nt, nl = rtp.reshard_cost(rtp.F32, UNEVEN_SHAPE, src, dst)
            torch.cuda.synchronize()
            rtp.reshard(ins, UNEVEN_SHAPE, src, dst, out=outs)
            torch.cuda.synchronize()
            order.append({"call": tname, "algorithmic_bytes": rd + wr, "launches": nl,
                          "forms": list(rtp.reshard_forms(rtp.F32, UNEVEN_SHAPE, src, dst))})
        print(json.dumps({"case": name, "calls": order}))
    elif kind == "reshard":
        mesh_name, idx, dt = det
        dtype, code = (torch.float32, rtp.F32) if dt == "f32" else (torch.bfloat16, rtp.BF16)
        _, src, dst, _ = sweep_specs(rtp, mesh_name)[idx]
        ins = [torch.randn(rtp.shard_shape(SWEEP_SHAPE, src, r), generator=gen, device="cuda").to(dtype)
               for r in range(src.num_ranks)]
        outs = [torch.empty(rtp.shard_shape(SWEEP_SHAPE, dst, r), dtype=dtype, device="cuda")
                for r in range(dst.num_ranks)]
        rd, wr, nt, nl = rtp.reshard_cost(code, SWEEP_SHAPE, src, dst)
        torch.cuda.synchronize()
        for _ in range(repeats):
            rtp.reshard(ins, SWEEP_SHAPE, src, dst, out=outs)
        torch.cuda.synchronize()
        print(json.dumps({"case": name, "algorithmic_bytes_per_launch": rd + wr, "launches_per_call": nl}))
    else:
        c = det
        M, K, F, N, P = c["M"], c["K"], c["F"], c["N"], c["P"]
        X = torch.randn((M, K), generator=gen, device="cuda").bfloat16()
        A = [(torch.randn((K, F // P), generator=gen, device="cuda") * 0.02).bfloat16() for _ in range(P)]
        B = [(torch.randn((F // P, N), generator=gen, device="cuda") * 0.02).bfloat16() for _ in range(P)]
        Y = [torch.empty((M, F // P), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
        Z = torch.empty((M, N), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        if kind == "mlp_backward":
            # training forward (2 launches) then backward (4 launches: dH, dX, dA, dB) per repeat
            dZ = torch.randn((M, N), generator=gen, device="cuda").bfloat16()
            for _ in range(repeats):
                _, Yt, H = rtp.tp_mlp_train_forward(X, A, B, Y=Y, Z=Z)
                rtp.tp_mlp_backward(X, A, B, H, Yt, dZ, mode=1)
            torch.cuda.synchronize()
            print(json.dumps({"case": name, "flops_per_gemm": [2 * M * K * F, 2 * M * F * N, 2 * M * N * F,
                                                               2 * M * F * K, 2 * K * M * F, 2 * F * M * N]}))
        elif kind == "mlp_library":
            # the fused MLP (2 launches), then the library GEMMs of the same
            # shapes (torch.mm: X [A_i] and Y [B_i], bf16 outputs, no GELU),
            # once each, inside the NVTX range "gemms"
            a_cat, b_cat = torch.cat(A, dim=1), torch.cat(B, dim=0)
            y_cat = torch.empty((M, F), dtype=torch.bfloat16, device="cuda")
            z_lib = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            torch.cuda.synchronize()
            torch.cuda.nvtx.range_push("gemms")
            rtp.tp_mlp(X, A, B, Y=Y, Z=Z, mode=1)
            torch.mm(X, a_cat, out=y_cat)
            torch.mm(y_cat, b_cat, out=z_lib)
            torch.cuda.nvtx.range_pop()
            torch.cuda.synchronize()
            print(json.dumps({"case": name, "flops_per_gemm": 2 * M * K * F}))
        else:
            for _ in range(repeats):
                rtp.tp_mlp(X, A, B, Y=Y, Z=Z, mode=1)
            torch.cuda.synchronize()
            print(json.dumps({"case": name, "flops_gemm1": 2 * M * K * F, "flops_gemm2": 2 * M * F * N}))
    assert rtp.device_error() == 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--profile-case", choices=sorted(PROFILE_CASES), default=None,
                    help="run one small fixed workload for an ncu capture and exit")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-library-gemm", action="store_true",
                    help="skip timing the fused MLP beside the library (cuBLAS) GEMMs after the timed region")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args.profile_case)
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus if args.gpus == 1 else 1)))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
