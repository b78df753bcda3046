#!/usr/bin/env python
"""Benchmark of causal context-parallel attention on one GB300.

Workload (default): ring attention forward, MHA, S=8192, H=32, D=128, bf16,
q/k/v ~ N(0,1) (seed 0), causal, P=8 virtual ranks, zigzag (dual-chunk-swap)
layout, fused ring schedule.  One step is one pass of the hot path over that
input: zigzag reorder of q, k, v into the ranks' layout, the ring attention
(one tcgen05 kernel walking every rank's key/value blocks in ring order, with
the log-sum-exp merge in its online softmax), and the restore of out and lse
to sequence order, which the attention's epilogue does by writing every output
row and lse column at its sequence position (each zigzag chunk is a run of
consecutive rows).  Inputs are resident in HBM when the timed region starts;
L2 is flushed between timed steps: 256 MiB are written, then another 256 MiB
read, so that the flush's own dirty lines are written back before the timed
region instead of inside it.

Prints ONE JSON line.  ``--impl reference`` times the CPU float64 oracle (the
correctness reference) on a bounded sample of the same workload instead.
Under torchrun with N>1 every rank runs the same workload on its own GPU
(replicas: the method has no cross-GPU step here) and rank 0 reports
N x work / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal CP-attn TFLOP/s (fwd, fwd+bwd) & permute GB/s, % of roofline, 1 GB300"
WORKLOAD = "ring_fwd_mha_s8192_h32_d128_bf16_p8_zigzag"
S, H, D, P = 8192, 32, 128, 8
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


def _r(x, sig: int = 4):
    """Floats rounded to `sig` significant digits, recursively (keeps the line short)."""
    if isinstance(x, float):
        return float(f"{x:.{sig}g}") if math.isfinite(x) else x
    if isinstance(x, dict):
        return {k: _r(v, sig) for k, v in x.items()}
    if isinstance(x, (list, tuple)):
        return [_r(v, sig) for v in x]
    return x


def causal_flop(S: int, H: int, D: int) -> float:
    """4*D FLOP per visible (query, key) pair per head (QK^T and PV)."""
    return 4.0 * D * H * (S * (S + 1) // 2)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    return ws, rank


def max_over_ranks(x: float, device=None) -> float:
    """The slowest rank's value (time-like numbers), identical on every rank;
    the input itself on one process."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flop_per_rank: float, world: int, ms: float) -> float:
    """Throughput of the whole job: every rank processed flop_per_rank in at most ms."""
    return world * flop_per_rank / (ms * 1e-3) / 1e12


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return dict(FALLBACK_PEAKS, bf16_tflops_sustained=1700.0, source="fallback")


def _traffic_record(kernel_key: str):
    """DRAM bytes per launch of a kernel from a committed ncu capture, or None
    when the kernel's source has changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path)).get(kernel_key)
    if not rec:
        return None
    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src):
        return None
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if h != rec.get("source_sha256_16"):
        return None
    return float(rec["bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms in the background."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(device_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.t_start = self.t_end = None

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def finish(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t_start - 1 <= r[0] <= self.t_end + 1] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3]) if v.lower() == "active"})
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


def _oracle_inputs(q, k, v):
    return (q.float().numpy().astype(np.float64), k.float().numpy().astype(np.float64),
            v.float().numpy().astype(np.float64))


def _oracle_rows(qs, ks, vs, n, rng):
    """Times the float64 oracle on n random query rows (all heads) against the full
    causal key range; returns (FLOP of those rows, seconds)."""
    import oracle

    rows = np.sort(rng.integers(0, S, size=n))
    t0 = time.perf_counter()
    oracle.attention(qs[rows], ks, vs, True, pos_q=rows, pos_k=np.arange(S))
    dt = time.perf_counter() - t0
    return 4.0 * D * H * float(np.sum(rows + 1)), dt


def host_info() -> dict:
    """The oracle timing host: CPUs in this process's affinity mask, all CPUs, and
    the BLAS numpy was built against (its thread pool runs the oracle's products)."""
    info = {"affinity_cpus": len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else None,
            "cpu_count": os.cpu_count(), "machine": platform.machine()}
    try:
        import numpy as np
        cfg = np.show_config(mode="dicts")
        blas = cfg.get("Build Dependencies", {}).get("blas", {})
        info["blas"] = f"{blas.get('name', '?')} {blas.get('version', '')}".strip()
    except Exception:  # older numpy: no dict form
        info["blas"] = "unknown"
    return info


def cpu_oracle_sample(q, k, v, target_s: float = 12.0):
    """Oracle throughput on a bounded sample sized to about target_s seconds.
    Returns (TFLOP/s, rows, seconds)."""
    qs, ks, vs = _oracle_inputs(q, k, v)
    rng = np.random.default_rng(123)
    _, dt = _oracle_rows(qs, ks, vs, 8, rng)
    n = int(max(8, min(4096, 8 * target_s / max(dt, 1e-3))))
    flop, dt = _oracle_rows(qs, ks, vs, n, rng)
    return flop / dt / 1e12, n, dt


def bench_reference(args):
    ws, rank = _dist()
    if rank != 0:
        return
    from synth import make_inputs

    q, k, v = make_inputs(S, H, H, D, torch.bfloat16, seed=0)
    qs, ks, vs = _oracle_inputs(q, k, v)
    rng = np.random.default_rng(123)
    # one calibration, then every step is the same bounded sample size (~90 s in all)
    _, dt8 = _oracle_rows(qs, ks, vs, 8, rng)
    per_step_s = min(1.0, 90.0 / max(1, args.steps + args.warmup))
    n = int(max(1, min(4096, 8 * per_step_s / max(dt8, 1e-3))))
    per_step = []
    for i in range(args.warmup + args.steps):
        flop, dt = _oracle_rows(qs, ks, vs, n, rng)
        if i >= args.warmup:
            per_step.append((flop / dt / 1e12, dt))
    value = statistics.mean(t for t, _ in per_step)
    ms = 1e3 * statistics.mean(d for _, d in per_step)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic N(0,1), seed 0",
        "config": {"workload": WORKLOAD, "S": S, "H": H, "D": D, "P": P, "reorder": "dual_chunk_swap"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} random query rows x {H} heads per step, full causal key range",
                         "host": host_info()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def bench_ours(args):
    import context_causal_attention_tcgen05_gb300 as cpa
    from synth import make_inputs

    ws, rank = _dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    cpa.load_library()  # raises when the library is missing: there is no fallback
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    q_h, k_h, v_h = make_inputs(S, H, H, D, torch.bfloat16, seed=0)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    q_re, k_re, v_re = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    out = torch.empty_like(q)
    lse = torch.empty(H, S, dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty(1, dtype=torch.float32, device=dev)

    def flush_l2():
        # write > L2, then read > L2: the written lines leave L2 (written back) before
        # the timed region, which then pays only for its own traffic
        flush.fill_(1.0)
        flush_sink.copy_(flush_rd.sum().view(1))

    layout = "zigzag"

    def step(ev):
        ev[0].record(stream)
        cpa.cp_ring_reorder_qkv(q, k, v, P, layout, q_re=q_re, k_re=k_re, v_re=v_re)
        ev[1].record(stream)
        # the ring writes out and lse at their sequence positions: the restore is done
        # by the attention's own output writes (every zigzag chunk is a run of rows)
        cpa.cp_ring_attention_reordered_to_seq(q_re, k_re, v_re, P, layout, out=out, lse=lse)
        ev[2].record(stream)
        ev[3].record(stream)

    launches_per_step = 2  # q/k/v reorder, attention (restore in its epilogue)
    mk = lambda: [torch.cuda.Event(enable_timing=True) for _ in range(4)]

    def timed(fn, reps):
        """Mean device time (ms) of fn over reps, L2 flushed before each rep."""
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            flush_l2()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            fn()
            b_.record(stream)
            ts.append((a_, b_))
        torch.cuda.synchronize()
        return statistics.mean(x.elapsed_time(y) for x, y in ts)

    def hbm_parts(reps):
        """GB/s of the HBM-bound kernels on their workload shapes (algorithmic bytes:
        every byte read once and written once)."""
        out = {}
        # LSE merge in fp32 at the ring shape (the stepwise ring's accumulator update)
        o1 = torch.randn(S, H, D, device=dev)
        o2 = torch.randn(S, H, D, device=dev)
        l1 = torch.randn(H, S, device=dev)
        l2 = torch.randn(H, S, device=dev)
        ms = timed(lambda: cpa.cp_lse_merge(o1, l1, o2, l2, out=o1, lse=l1), reps)
        nbytes = 3 * o1.numel() * 4 + 3 * l1.numel() * 4
        out["lse_merge_f32_s8192_h32_d128"] = {"ms": ms, "gbs": nbytes / (ms * 1e-3) / 1e9, "bytes": nbytes}
        del o1, o2
        b1 = torch.randn(S, H, D, device=dev).to(torch.bfloat16)
        b2 = torch.randn(S, H, D, device=dev).to(torch.bfloat16)
        ms = timed(lambda: cpa.cp_lse_merge(b1, l1, b2, l2, out=b1, lse=l1), reps)
        nbytes = 3 * b1.numel() * 2 + 3 * l1.numel() * 4
        out["lse_merge_bf16_s8192_h32_d128"] = {"ms": ms, "gbs": nbytes / (ms * 1e-3) / 1e9, "bytes": nbytes}
        del b1, b2, l1, l2
        # the same merges at the GQA ring shape (S=65536, H=32)
        S4 = 65536
        l1 = torch.randn(H, S4, device=dev)
        l2 = torch.randn(H, S4, device=dev)
        for name, dt, esz in (("f32", torch.float32, 4), ("bf16", torch.bfloat16, 2)):
            c1 = torch.randn(S4, H, D, device=dev).to(dt)
            c2 = torch.randn(S4, H, D, device=dev).to(dt)
            ms = timed(lambda: cpa.cp_lse_merge(c1, l1, c2, l2, out=c1, lse=l1), reps)
            nbytes = 3 * c1.numel() * esz + 3 * l1.numel() * 4
            out[f"lse_merge_{name}_s65536_h32_d128"] = {"ms": ms, "gbs": nbytes / (ms * 1e-3) / 1e9,
                                                       "bytes": nbytes}
            del c1, c2
        del l1, l2
        # Ulysses seq2head + head2seq at S=32768, H=32, D=128, P=16 (bf16)
        Su, Pu = 32768, 16
        x = torch.randn(Su, H, D, device=dev).to(torch.bfloat16)
        y = torch.empty(Pu, Su, H // Pu, D, dtype=torch.bfloat16, device=dev)
        ms1 = timed(lambda: cpa.cp_ulysses_seq2head(x, Pu, y=y), reps)
        ms2 = timed(lambda: cpa.cp_ulysses_head2seq(y, Pu, x=x), reps)
        nbytes = 2 * x.numel() * 2
        out["ulysses_seq2head_s32768_h32_d128_p16"] = {"ms": ms1, "gbs": nbytes / (ms1 * 1e-3) / 1e9, "bytes": nbytes}
        out["ulysses_head2seq_s32768_h32_d128_p16"] = {"ms": ms2, "gbs": nbytes / (ms2 * 1e-3) / 1e9, "bytes": nbytes}
        del x, y
        return out

    def ulysses_fwd(reps):
        """Ulysses forward at S=32768, H=32, D=128, P=16 (2 heads per virtual rank):
        the whole driver (seq2head of q, k, v; attention, whose epilogue writes out
        in sequence layout, i.e. does the head2seq) and its three permutes on their
        own, device-resident inputs."""
        Su, Pu = 32768, 16
        qu, ku, vu = (t.to(dev) for t in make_inputs(Su, H, H, D, torch.bfloat16, 0))
        ou, lu = torch.empty_like(qu), torch.empty(H, Su, dtype=torch.float32, device=dev)
        wu = torch.empty(cpa.cp_workspace_size("ulysses_fwd", Su, H, H, D, torch.bfloat16, Pu),
                         dtype=torch.uint8, device=dev)
        y = [torch.empty(Pu, Su, H // Pu, D, dtype=torch.bfloat16, device=dev) for _ in range(3)]
        total = timed(lambda: cpa.cp_ulysses_attention(qu, ku, vu, Pu, out=ou, lse=lu, workspace=wu), reps)

        def perms():
            for x, yy in zip((qu, ku, vu), y):
                cpa.cp_ulysses_seq2head(x, Pu, y=yy)

        perm = timed(perms, reps)
        f = causal_flop(Su, H, D)
        nbytes = 3 * 2 * qu.numel() * 2
        # backward through the public driver (dO ~ N(0,1), seed 1)
        dou = torch.randn(qu.shape, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).to(dev)
        wb = torch.empty(cpa.cp_workspace_size("ulysses_bwd", Su, H, H, D, torch.bfloat16, Pu),
                         dtype=torch.uint8, device=dev)
        dq, dk, dv = torch.empty_like(qu), torch.empty_like(ku), torch.empty_like(vu)
        bwd = timed(lambda: cpa.cp_ulysses_attention_bwd(qu, ku, vu, ou, lu, dou, Pu, dq=dq, dk=dk, dv=dv,
                                                         workspace=wb), reps)
        del qu, ku, vu, ou, lu, wu, y, dou, wb, dq, dk, dv
        return {"workload": "ulysses_fwd_s32768_h32_d128_bf16_p16", "flop": f, "driver_ms": total,
                "driver_tflops": f / (total * 1e-3) / 1e12, "permute_ms": perm,
                "permute_gbs": nbytes / (perm * 1e-3) / 1e9,
                "attention_ms": total - perm, "attention_tflops": f / ((total - perm) * 1e-3) / 1e12,
                "bwd_driver_ms": bwd, "bwd_tflops": 2.5 * f / (bwd * 1e-3) / 1e12,
                "fwd_bwd_tflops": 3.5 * f / ((total + bwd) * 1e-3) / 1e12}

    def varlen_fwd(reps):
        """Packed varlen ring forward at S=131072, Hq=32, Hkv=8, D=128, P=8, documents
        of U[512, 16384] tokens (seed 0): attention phase on reordered inputs per
        strategy; FLOP count only the visible (same-document, causal) pairs."""
        from synth import cu_seqlens_from_lengths, doc_lengths

        Sv, Hqv, Hkvv, Pv = 131072, 32, 8, 8
        cu = cu_seqlens_from_lengths(doc_lengths(Sv, 512, 16384, seed=0))
        lens = np.diff(cu).astype(np.int64)
        pairs = float(np.sum(lens * (lens + 1) // 2))
        f = 4.0 * D * Hqv * pairs
        # visible pairs of each virtual rank's queries (every key of the sequence is visited)
        pos = np.arange(Sv)
        start = np.repeat(cu[:-1], lens)
        vis = (pos - start + 1).astype(np.float64)
        C = Sv // (2 * Pv)
        out = {"workload": "packed_varlen_fwd_s131072_hq32_hkv8_d128_bf16_p8", "docs": int(len(lens)),
               "flop": f, "visible_pairs_per_head": pairs}
        qv, kv, vv = (t.to(dev) for t in make_inputs(Sv, Hqv, Hkvv, D, torch.bfloat16, 0))
        cu_d = torch.from_numpy(cu).to(dev)
        for layout in ("striped", "zigzag"):
            if layout == "striped":
                per_rank = [float(vis[r::Pv].sum()) for r in range(Pv)]
                reo = lambda x: cpa.cp_striped_reorder(x, Pv)
            else:
                per_rank = [float(vis[r * C:(r + 1) * C].sum() + vis[(2 * Pv - 1 - r) * C:(2 * Pv - r) * C].sum())
                            for r in range(Pv)]
                reo = lambda x: cpa.cp_zigzag_reorder(x, Pv)
            qr, kr, vr = reo(qv), reo(kv), reo(vv)
            o = torch.empty_like(qr)
            l = torch.empty(Hqv, Sv, dtype=torch.float32, device=dev)
            ms = timed(lambda: cpa.cp_ring_attention_reordered(qr, kr, vr, Pv, layout, "fused", cu_seqlens=cu_d,
                                                               out=o, lse=l), reps)
            out[layout] = {"attention_ms": ms, "tflops": f / (ms * 1e-3) / 1e12,
                           "rank_visible_pairs": per_rank,
                           "imbalance_max_over_mean": max(per_rank) / (sum(per_rank) / Pv)}
            del qr, kr, vr, o, l
        del qv, kv, vv, cu_d
        return out

    def gqa_fwd_bwd(n_steps):
        """fwd and fwd+bwd of the GQA ring workload (S=65536, Hq=32, Hkv=8, D=128,
        P=4, zigzag) through the public drivers, device-resident inputs."""
        S4, Hq4, Hkv4, D4, P4 = 65536, 32, 8, 128, 4
        q4, k4, v4, do4 = (t.to(dev) for t in make_inputs(S4, Hq4, Hkv4, D4, torch.bfloat16, 0, True))
        o4, l4 = torch.empty_like(q4), torch.empty(Hq4, S4, dtype=torch.float32, device=dev)
        dq4, dk4, dv4 = torch.empty_like(q4), torch.empty_like(k4), torch.empty_like(v4)
        wf = torch.empty(cpa.cp_workspace_size("ring_fwd", S4, Hq4, Hkv4, D4, torch.bfloat16, P4),
                         dtype=torch.uint8, device=dev)
        wb = torch.empty(cpa.cp_workspace_size("ring_bwd", S4, Hq4, Hkv4, D4, torch.bfloat16, P4),
                         dtype=torch.uint8, device=dev)

        def one(ev=None):
            if ev:
                ev[0].record(stream)
            cpa.cp_ring_attention(q4, k4, v4, P4, "zigzag", "fused", out=o4, lse=l4, workspace=wf)
            if ev:
                ev[1].record(stream)
            cpa.cp_ring_attention_bwd(q4, k4, v4, o4, l4, do4, P4, "zigzag", dq=dq4, dk=dk4, dv=dv4,
                                      workspace=wb)
            if ev:
                ev[2].record(stream)

        for _ in range(2):
            one()
        torch.cuda.synchronize()
        evs = []
        for _ in range(n_steps):
            flush_l2()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            one(ev)
            evs.append(ev)
        torch.cuda.synchronize()
        fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
        bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
        f = causal_flop(S4, Hq4, D4)
        del q4, k4, v4, do4, o4, l4, dq4, dk4, dv4, wf, wb
        return {"workload": "gqa_ring_fwd_bwd_s65536_hq32_hkv8_d128_bf16_p4_zigzag",
                "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "fwd_tflops": f / (fwd_ms * 1e-3) / 1e12,
                "bwd_tflops": 2.5 * f / (bwd_ms * 1e-3) / 1e12,
                "fwd_bwd_tflops": 3.5 * f / ((fwd_ms + bwd_ms) * 1e-3) / 1e12,
                "flop_fwd": f, "flop_bwd": 2.5 * f, "steps": n_steps}
    for _ in range(args.warmup):
        step(mk())
    torch.cuda.synchronize()
    st = cpa.cp_check_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st}: {cpa.cp_last_error()}")

    sampler = ClockSampler(torch.cuda.current_device())
    time.sleep(0.6)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.mark_start()
    events = []
    for _ in range(args.steps):
        flush_l2()  # write > L2, then read > L2, between steps (outside the events)
        ev = mk()
        step(ev)
        events.append(ev)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    fb = gqa_fwd_bwd(args.fwd_bwd_steps) if args.fwd_bwd_steps > 0 else None
    hbm = hbm_parts(max(5, min(args.steps, 20)))
    uly = ulysses_fwd(5) if args.fwd_bwd_steps > 0 else None
    vlen = varlen_fwd(5) if args.fwd_bwd_steps > 0 else None
    sampler.mark_end()
    clocks = sampler.finish()
    st = cpa.cp_check_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st}: {cpa.cp_last_error()}")

    step_ms = [e[0].elapsed_time(e[3]) for e in events]
    attn_ms = [e[1].elapsed_time(e[2]) for e in events]
    perm_ms = [e[0].elapsed_time(e[1]) + e[2].elapsed_time(e[3]) for e in events]
    mean_step = max_over_ranks(statistics.mean(step_ms), dev)
    flop = causal_flop(S, H, D)
    value = whole_job_tflops(flop, ws, mean_step)
    attn_mean = statistics.mean(attn_ms)
    achieved = flop / (attn_mean * 1e-3) / 1e12
    tensor_bytes = S * H * D * 2
    perm_bytes = 3 * 2 * tensor_bytes  # q, k, v read and written once
    perm_gbs = perm_bytes / (statistics.mean(perm_ms) * 1e-3) / 1e9

    # end to end through the public one-call driver with host buffers: every step
    # copies its q, k, v from pinned host memory and reads out and lse back.  Steps
    # are independent, so they are pipelined as a user would run them: two device
    # buffer sets, copy-in / compute / copy-out on three streams (step i's copy-in
    # overlaps step i-1's compute and step i-2's copy-out).  The inputs of a step
    # (192 MiB) exceed L2, so no flush is needed between steps.
    q_p, k_p, v_p = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
    wsz = cpa.cp_workspace_size("ring_fwd", S, H, H, D, torch.bfloat16, P, "fused")
    nb = 2
    bufs = [dict(q=torch.empty_like(q), k=torch.empty_like(k), v=torch.empty_like(v), o=torch.empty_like(q),
                 l=torch.empty_like(lse), w=torch.empty(wsz, dtype=torch.uint8, device=dev),
                 op=torch.empty(out.shape, dtype=out.dtype).pin_memory(),
                 lp=torch.empty(lse.shape, dtype=lse.dtype).pin_memory()) for _ in range(nb)]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = [dict(inp=torch.cuda.Event(), cmp=torch.cuda.Event(), out=torch.cuda.Event()) for _ in range(nb)]

    def e2e_run(n_steps, start_ev=None, end_ev=None):
        torch.cuda.synchronize()
        if start_ev is not None:
            start_ev.record(s_in)
            s_cmp.wait_stream(s_in)
            s_out.wait_stream(s_in)
        for i in range(n_steps):
            bb, e = bufs[i % nb], ev[i % nb]
            if i >= nb:
                s_in.wait_event(e["cmp"])  # the compute that read this buffer set is done
            with torch.cuda.stream(s_in):
                bb["q"].copy_(q_p, non_blocking=True)
                bb["k"].copy_(k_p, non_blocking=True)
                bb["v"].copy_(v_p, non_blocking=True)
            e["inp"].record(s_in)
            s_cmp.wait_event(e["inp"])
            if i >= nb:
                s_cmp.wait_event(e["out"])  # the copy-out of this buffer set's last result is done
            cpa.cp_ring_attention(bb["q"], bb["k"], bb["v"], P, layout, "fused", out=bb["o"], lse=bb["l"],
                                  workspace=bb["w"], stream=s_cmp)
            e["cmp"].record(s_cmp)
            s_out.wait_event(e["cmp"])
            with torch.cuda.stream(s_out):
                bb["op"].copy_(bb["o"], non_blocking=True)
                bb["lp"].copy_(bb["l"], non_blocking=True)
            e["out"].record(s_out)
        if end_ev is not None:
            s_out.wait_stream(s_in)
            s_out.wait_stream(s_cmp)
            end_ev.record(s_out)
        torch.cuda.synchronize()

    e2e_run(max(3, args.warmup))
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(args.steps, ea, eb)
    e2e_mean = ea.elapsed_time(eb) / args.steps
    # the same step without overlap (one stream, one step at a time), for reference
    ser = []
    for i in range(min(args.steps, 20)):
        bb = bufs[0]
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        bb["q"].copy_(q_p, non_blocking=True)
        bb["k"].copy_(k_p, non_blocking=True)
        bb["v"].copy_(v_p, non_blocking=True)
        cpa.cp_ring_attention(bb["q"], bb["k"], bb["v"], P, layout, "fused", out=bb["o"], lse=bb["l"],
                              workspace=bb["w"])
        bb["op"].copy_(bb["o"], non_blocking=True)
        bb["lp"].copy_(bb["l"], non_blocking=True)
        b_.record(stream)
        ser.append((a_, b_))
    torch.cuda.synchronize()
    e2e_serial = statistics.mean(x.elapsed_time(y) for x, y in ser)
    st = cpa.cp_check_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st}: {cpa.cp_last_error()}")
    e2e_mean = max_over_ranks(e2e_mean, dev)
    e2e_value = whole_job_tflops(flop, ws, e2e_mean)

    if rank == 0:
        peaks = _peaks()
        peak = peaks["bf16_tflops"]
        traffic = _traffic_record("attn_fwd_tc")
        cpu_tf, cpu_rows, cpu_s = (None, 0, 0.0)
        if not args.no_cpu_baseline:
            cpu_tf, cpu_rows, cpu_s = cpu_oracle_sample(q_h, k_h, v_h)
        cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": mean_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic N(0,1), seed 0",
            "config": {"workload": WORKLOAD, "S": S, "H": H, "D": D, "P": P, "reorder": "dual_chunk_swap",
                       "ring_mode": "fused", "l2": "flushed between timed steps (256 MiB write, then 256 MiB read)"},
            "gpu_launches": launches_per_step * args.steps,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": "attn_fwd_tc (ring, fused)", "peak_source": peaks["source"] + " burst bf16"},
            "e2e": _r({"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": 3 * tensor_bytes,
                       "d2h_bytes_per_step": tensor_bytes + S * H * 4, "ms_per_step": e2e_mean,
                       "pipeline": "2 buffer sets; copy-in, compute, copy-out on 3 streams",
                       "serial_ms_per_step": e2e_serial,
                       "serial_value": flop / (e2e_serial * 1e-3) / 1e12}),
            "clocks": clocks,
        }
        if cpu_tf is not None:
            line["cpu_baseline"] = {"value": cpu_tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                    "sample": f"{cpu_rows} random query rows x {H} heads, full causal key "
                                              f"range ({cpu_s:.1f} s of float64 CPU work)",
                                    "host": host_info()}
        # the other workloads' parts, the fwd+bwd of the largest one last
        line["parts"] = _r({"attention_ms": attn_mean, "attention_tflops": achieved,
                            "permute_ms": statistics.mean(perm_ms), "permute_gbs": perm_gbs,
                            "permute_frac_of_hbm": perm_gbs / peaks["hbm_gbs"]})
        line["hbm_kernels"] = _r({k: {"ms": v["ms"], "gbs": v["gbs"], "frac_of_hbm": v["gbs"] / peaks["hbm_gbs"]}
                                  for k, v in hbm.items()})
        if uly is not None:
            line["ulysses_fwd"] = _r(dict(uly, frac_of_peak=uly["attention_tflops"] / peak,
                                          permute_frac_of_hbm=uly["permute_gbs"] / peaks["hbm_gbs"],
                                          fwd_bwd_frac_of_peak=uly["fwd_bwd_tflops"] / peak))
        if vlen is not None:
            for lay in ("striped", "zigzag"):
                vlen[lay].pop("rank_visible_pairs", None)
            line["varlen_fwd"] = _r(dict(vlen, frac_of_peak={k: vlen[k]["tflops"] / peak
                                                             for k in ("striped", "zigzag")}))
        if fb is not None:
            line["fwd_bwd"] = _r(dict(fb, fwd_frac_of_peak=fb["fwd_tflops"] / peak,
                                      bwd_frac_of_peak=fb["bwd_tflops"] / peak,
                                      frac_of_peak=fb["fwd_bwd_tflops"] / peak))
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def profile_case(args) -> int:
    """Runs one hot-path case a few times on cuda:0, for profiler captures (ncu):
    ring_fwd (reordered inputs, fused ring: one attention launch per rep), ring_bwd
    (ring backward), permute (zigzag reorder of q), reorder_qkv (q, k, v in one
    launch), ulysses (seq2head of q), merge (in-place fp32 or bf16 LSE merge of two
    [S, Hq, D] partial outputs).  Inputs are N(0,1) bf16 from the seeded
    generators.  Returns non-zero if the library reports an error."""
    import context_causal_attention_tcgen05_gb300 as cpa
    from synth import make_inputs

    a = args
    torch.cuda.set_device(0)
    cpa.load_library()
    q, k, v, do = (t.cuda() for t in make_inputs(a.S, a.Hq, a.Hkv, a.D, torch.bfloat16, 0, True))
    cu_d = None
    if a.docs:
        from synth import cu_seqlens_from_lengths, doc_lengths
        cu_d = torch.from_numpy(cu_seqlens_from_lengths(doc_lengths(a.S, 512, 16384, seed=0))).cuda()
    if a.profile_case == "ring_fwd":
        reo = {"zigzag": cpa.cp_zigzag_reorder, "striped": cpa.cp_striped_reorder}.get(a.layout)
        qr, kr, vr = (reo(x, a.P) if reo else x for x in (q, k, v))
        for _ in range(a.reps):
            cpa.cp_ring_attention_reordered(qr, kr, vr, a.P, a.layout, "fused", cu_seqlens=cu_d)
    elif a.profile_case == "ring_bwd":
        o, l = cpa.cp_ring_attention(q, k, v, a.P, a.layout, "fused", cu_seqlens=cu_d)
        ws = torch.empty(cpa.cp_workspace_size("ring_bwd", a.S, a.Hq, a.Hkv, a.D, q.dtype, a.P),
                         dtype=torch.uint8, device=q.device)
        for _ in range(a.reps):
            cpa.cp_ring_attention_bwd(q, k, v, o, l, do, a.P, a.layout, cu_seqlens=cu_d, workspace=ws)
    elif a.profile_case == "merge":
        g = torch.Generator(device="cuda").manual_seed(1)
        dt = torch.bfloat16 if a.merge_dtype == "bf16" else torch.float32
        o1 = torch.randn(a.S, a.Hq, a.D, device="cuda", generator=g).to(dt)
        o2 = torch.randn(a.S, a.Hq, a.D, device="cuda", generator=g).to(dt)
        l1 = torch.randn(a.Hq, a.S, device="cuda", generator=g)
        l2 = torch.randn(a.Hq, a.S, device="cuda", generator=g)
        for _ in range(a.reps):
            cpa.cp_lse_merge(o1, l1, o2, l2, out=o1, lse=l1)
    elif a.profile_case == "reorder_qkv":
        ys = [torch.empty_like(x) for x in (q, k, v)]
        for _ in range(a.reps):
            cpa.cp_ring_reorder_qkv(q, k, v, a.P, a.layout, q_re=ys[0], k_re=ys[1], v_re=ys[2])
    elif a.profile_case == "permute":
        y = torch.empty_like(q)
        for _ in range(a.reps):
            cpa.cp_zigzag_reorder(q, a.P, y=y)
    else:  # ulysses
        y = torch.empty(a.P, a.S, a.Hq // a.P, a.D, dtype=q.dtype, device=q.device)
        for _ in range(a.reps):
            cpa.cp_ulysses_seq2head(q, a.P, y=y)
    torch.cuda.synchronize()
    st = cpa.cp_check_device_status()
    if st != 0:
        print("device status", st, cpa.cp_last_error(), file=sys.stderr)
        return 1
    print("ok")
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--fwd-bwd-steps", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    # one profiler case instead of the benchmark (see profile_case)
    ap.add_argument("--profile-case", choices=["ring_fwd", "ring_bwd", "permute", "reorder_qkv", "ulysses",
                                               "merge"])
    ap.add_argument("--S", type=int, default=8192)
    ap.add_argument("--Hq", type=int, default=32)
    ap.add_argument("--Hkv", type=int, default=32)
    ap.add_argument("--D", type=int, default=128)
    ap.add_argument("--P", type=int, default=8)
    ap.add_argument("--layout", default="zigzag")
    ap.add_argument("--docs", action="store_true", help="pack documents (lengths U[512, 16384], seed 0)")
    ap.add_argument("--merge-dtype", choices=["f32", "bf16"], default="f32")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    if args.profile_case:
        sys.exit(profile_case(args))
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
