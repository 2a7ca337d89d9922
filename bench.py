"""Benchmark of one Ulysses attention layer step on GB300.

A step is the whole hot path over one batch of synthetic input:
  seq->head swap of Q, K, V  ->  attention forward  ->  head->seq swap of O
  ->  seq->head swap of dO  ->  attention backward  ->  head->seq swap of dQ, dK, dV
through the library's C ABI (via its Python binding).

Default workload: Qwen3-4B-shaped attention at long context -- batch 1,
N = 65536 tokens, P = 4 virtual ranks, 32 query / 8 KV heads, head_dim 128,
bf16, causal, Q/K/V/dO ~ N(0, 1).

Printed JSON line (rank 0): value = attention fwd+bwd TFLOP/s of the whole
step, FLOPs counted algorithmically over the allowed (i, j) pairs only
(forward 4*d*Hq*pairs; backward 2.5x forward, i.e. five products per pair
including the recomputed scores), divided by the step's device time.

--gpus N under torchrun runs N independent replicas (the method's data path
is emulated on one GPU; there is no cross-GPU exchange), weak scaling.
--impl reference times the fp64 CPU oracle on bounded samples of the same
workload (the reference arm of this benchmark).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal attn fwd+bwd TFLOP/s (% bf16 TC peak) & tokens/s; layout-swap GB/s"
UNIT = "TFLOP/s"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def _pairs(N: int, cu) -> int:
    if cu is None:
        return N * (N + 1) // 2
    import numpy as np
    L = np.diff(np.asarray(cu, dtype=np.int64))
    return int((L * (L + 1) // 2).sum())


def _workload(name, seq_len=None):
    import dataclasses
    from ulysses_inputs import WORKLOADS, cu_seqlens_from_lengths, doc_lengths
    w = WORKLOADS[name]
    if seq_len:
        w = dataclasses.replace(w, N=int(seq_len))
    cu = cu_seqlens_from_lengths(doc_lengths(w.N, w.P, seed=3)) if w.packed_docs else None
    return w, cu


def _config(w, args, world):
    """The workload description both arms print (the same keys and values, so
    that the two lines can be matched)."""
    es = 2 if w.dtype == "bf16" else 4
    in_bytes = w.P * w.B * (w.N // w.P) * (2 * w.Hq + 2 * w.Hkv) * w.d * es
    return {"workload": args.workload + (f" (N overridden to {w.N})" if args.seq_len else ""), "B": w.B,
            "N": w.N, "P": w.P, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "causal": w.causal,
            "head_shards_timed": w.shards_timed, "packed_docs": w.packed_docs,
            "l2": "no flush: inputs larger than L2 (Q,K,V,dO %.2f GiB per step)" % (in_bytes / 2**30),
            "parallelism": f"replicas x{world} (virtual P={w.P} inside each GPU)"}


def _flops(w, cu):
    fwd = 4.0 * w.d * (w.Hp * w.shards_timed) * w.B * _pairs(w.N, cu)
    return fwd, 2.5 * fwd


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, log_dir: str = ""):
        import tempfile
        self.index = index
        self.proc = None
        self.path = os.path.join(log_dir or tempfile.gettempdir(), f"clocks_rank{index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[3], parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# -------------------------------------------------------- multi-rank logic
def max_over_ranks(value: float, dist, device=None) -> float:
    """The slowest rank's time (all ranks of a replica run do equal work)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_throughput(world: int, flops_per_rank_step: float, ms_per_step: float) -> float:
    """TFLOP/s of all ranks together: every replica processes one step per
    ms_per_step (the max over ranks)."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


# ------------------------------------------------------------- our arm
def pipelined_steps(n_steps, stream, up, down, step, sets_in, sets_out, result_of, h_in_of, h_out_of,
                    one_output_set=False):
    """Run `n_steps` calls of `step` as a stream of batches, with every step's
    inputs uploaded from and results read back to pinned host memory.

    Two device input sets alternate: the upload of step i+1 (stream `up`) and
    the read-back of step i-1 (stream `down`) run while step i computes on
    `stream`.  A step starts once its Q, K, V are in; dO, first read after the
    forward, follows them (`before_do`); its O is read back while its backward
    runs (`after_o`), the rest once the step is done.  `h_in_of(i)` and
    `h_out_of(i)` give step i's host tensors, `result_of(i)` the device tensors
    its read-back copies; with `one_output_set` every step writes the same
    device outputs.  Returns the (start, end) timing events."""
    import torch
    ev_in, ev_do, ev_o, ev_done, ev_out = ([torch.cuda.Event() for _ in range(n_steps)] for _ in range(5))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up.wait_event(e0)
    down.wait_event(e0)

    def upload(i):
        with torch.cuda.stream(up):
            if i >= 2:
                up.wait_event(ev_done[i - 2])  # step i-2 has consumed this input set
            hin = h_in_of(i)
            for dx, hx in zip(sets_in[i % 2][:3], hin[:3]):
                dx.copy_(hx, non_blocking=True)
            ev_in[i].record(up)  # Q, K, V
            sets_in[i % 2][3].copy_(hin[3], non_blocking=True)
            ev_do[i].record(up)

    def read_back_o(i):
        ev_o[i].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(ev_o[i])
            h_out_of(i)[0].copy_(result_of(i)[0], non_blocking=True)

    def read_back(i):
        with torch.cuda.stream(down):
            down.wait_event(ev_done[i])
            for hx, dx in zip(h_out_of(i)[1:], result_of(i)[1:]):
                hx.copy_(dx, non_blocking=True)
            ev_out[i].record(down)

    upload(0)
    for i in range(n_steps):
        if i + 1 < n_steps:
            upload(i + 1)
        stream.wait_event(ev_in[i])
        if i >= 2:
            stream.wait_event(ev_out[i - 2])  # step i-2's results are out of this output set
        if one_output_set and i >= 1:
            stream.wait_event(ev_out[i - 1])
        step(ins=sets_in[i % 2], outs_seq=sets_out[i % 2], after_o=lambda: read_back_o(i),
             before_do=lambda: stream.wait_event(ev_do[i]))
        ev_done[i].record(stream)
        read_back(i)
    stream.wait_event(ev_out[n_steps - 1])
    e1.record(stream)
    return e0, e1


class Layer:
    """Device buffers and the step of one workload: the seq-layout inputs,
    the head-layout working tensors, the seq-layout outputs and the
    attention workspaces, all resident in HBM."""

    def __init__(self, uly, w, cu, dev, seed):
        import torch
        from ulysses_inputs import draw_seq_inputs
        self.uly, self.w, self.cu, self.dev = uly, w, cu, dev
        P, S, B, N, d = w.P, w.shards_timed, w.B, w.N, w.d
        seq = draw_seq_inputs(w, seed=seed, device="cuda")
        self.ins = (seq["q"], seq["k"], seq["v"], seq["dout"])
        bt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        E = lambda *s: torch.empty(*s, dtype=bt, device=dev)
        self.qh, self.kh, self.vh, self.doh = (E(P, B, N, w.Hp, d), E(P, B, N, w.Hkvp, d), E(P, B, N, w.Hkvp, d),
                                               E(P, B, N, w.Hp, d))
        self.oh, self.dqh, self.dkh, self.dvh = (E(S, B, N, w.Hp, d), E(S, B, N, w.Hp, d), E(S, B, N, w.Hkvp, d),
                                                 E(S, B, N, w.Hkvp, d))
        self.lse = torch.empty(S, B, w.Hp, N, dtype=torch.float32, device=dev)
        self.outs = (E(P, B, N // P, w.Hq, d), E(P, B, N // P, w.Hq, d), E(P, B, N // P, w.Hkv, d),
                     E(P, B, N // P, w.Hkv, d))
        nd = 0 if cu is None else len(cu) - 1
        self.ws_f = torch.empty(uly.ulysses_attn_workspace_size(B, N, w.Hp, w.Hkvp, d, S, nd, False, bt),
                                dtype=torch.uint8, device=dev)
        self.ws_b = torch.empty(uly.ulysses_attn_workspace_size(B, N, w.Hp, w.Hkvp, d, S, nd, True, bt),
                                dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream()
        # the 1M workload times one head shard; the swaps back need all shards
        self.full = S == P

    @property
    def launches_per_step(self) -> int:
        # swaps: Q/K/V in one launch, O back with dO in, dQ/dK/dV back (dO alone
        # when only some shards are timed); forward 1; backward 3 (pre-pass,
        # main, dQ conversion)
        return (3 if self.full else 2) + 1 + 3

    def step(self, ev=None, ins=None, outs_seq=None, after_o=None, before_do=None):
        """One layer step on the inputs `ins` = (q, k, v, dO) in the seq layout,
        writing (O, dQ, dK, dV) in the seq layout to `outs_seq`.  `after_o` is
        called once O is final, `before_do` before dO is first read."""
        uly, w, cu, P, S = self.uly, self.w, self.cu, self.w.P, self.w.shards_timed
        q, k, v, do = ins if ins is not None else self.ins
        o_seq, dq_seq, dk_seq, dv_seq = outs_seq if outs_seq is not None else self.outs
        qh, kh, vh, doh, oh, dqh, dkh, dvh = (self.qh, self.kh, self.vh, self.doh, self.oh, self.dqh, self.dkh,
                                              self.dvh)

        def mark(i):
            if ev is not None:
                ev[i].record(self.stream)
        mark(0)
        uly.ulysses_swap_batch([(q, qh, True), (k, kh, True), (v, vh, True)], P)
        mark(1)
        uly.ulysses_attn_fwd(qh[:S], kh[:S], vh[:S], oh, self.lse, causal=w.causal, cu_seqlens=cu,
                             workspace=self.ws_f)
        mark(2)
        if before_do is not None:
            before_do()
        if self.full:
            uly.ulysses_swap_batch([(oh, o_seq, False), (do, doh, True)], P)
        else:
            uly.ulysses_seq_to_head(do, doh, P)
        if after_o is not None:
            after_o()
        mark(3)
        uly.ulysses_attn_bwd(qh[:S], kh[:S], vh[:S], oh, self.lse, doh[:S], dqh, dkh, dvh, causal=w.causal,
                             cu_seqlens=cu, workspace=self.ws_b)
        mark(4)
        if self.full:
            uly.ulysses_swap_batch([(dqh, dq_seq, False), (dkh, dk_seq, False), (dvh, dv_seq, False)], P)
        mark(5)

    def swap_bytes(self) -> int:
        b = 2 * sum(x.numel() * x.element_size() for x in self.ins)
        if self.full:
            b += 2 * sum(x.numel() * x.element_size() for x in (self.oh, self.dqh, self.dkh, self.dvh))
        return b

    def time(self, steps, warmup, barrier, check):
        """Warm-up, then `steps` timed steps between barriers; returns the
        elapsed device ms and the mean ms of the five phases."""
        import torch
        for _ in range(warmup):
            self.step()
        barrier()
        check("after warm-up")
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(steps)]
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        barrier()
        t0.record(self.stream)
        for i in range(steps):
            self.step(evs[i])
        t1.record(self.stream)
        barrier()
        check("in the timed region")
        phase = [[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(5)] for i in range(steps)]
        return t0.elapsed_time(t1), [statistics.mean(p[j] for p in phase) for j in range(5)]


def _rates(w, cu, layer, ms, ph, tc_sus, hbm):
    fwd_flops, bwd_flops = _flops(w, cu)
    step_flops = fwd_flops + bwd_flops
    swap_ms = ph[0] + ph[2] + ph[4]  # phases 0, 2 and 4 hold every swap
    sb = layer.swap_bytes() if layer.full else 2 * sum(
        x.numel() * x.element_size() for x in layer.ins)
    fb = step_flops / ((ph[1] + ph[3]) * 1e-3) / 1e12
    return {
        "ms_per_step": round(ms, 3), "value": round(step_flops / (ms * 1e-3) / 1e12, 2),
        "tokens_per_s": round(w.B * w.N / (ms * 1e-3), 1),
        "attn_fwd_tflops": round(fwd_flops / (ph[1] * 1e-3) / 1e12, 1),
        "attn_bwd_tflops": round(bwd_flops / (ph[3] * 1e-3) / 1e12, 1),
        "attn_fwd_bwd_tflops": round(fb, 1), "attn_fwd_bwd_frac_of_bf16_peak": round(fb / tc_sus, 3),
        "swap_gbps": round(sb / (swap_ms * 1e-3) / 1e9, 1),
        "swap_frac_of_hbm": round(sb / (swap_ms * 1e-3) / 1e9 / hbm, 3),
        "phase_ms": {"swap_qkv": round(ph[0], 3), "attn_fwd": round(ph[1], 3),
                     "swap_o_and_do": round(ph[2], 3), "attn_bwd": round(ph[3], 3),
                     "swap_dq_dk_dv": round(ph[4], 3)}}


# the other workloads timed beside the headline one: (name, steps, warm-up)
OTHER_WORKLOADS = (("qwen3_4b_n8192", 10, 3), ("packed_docs_n32768", 10, 3), ("tiny_fp32_n256", 10, 3),
                   ("single_shard_n1m", 1, 1))


def run_ours(args, rank, world, dist):
    import torch
    import long_context_sequence_head_gb300 as uly

    uly.load(build_if_missing=True)
    w, cu = _workload(args.workload, args.seq_len)
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    P, S, B, N, d = w.P, w.shards_timed, w.B, w.N, w.d
    layer = Layer(uly, w, cu, dev, args.seed + rank)
    q, k, v, do = layer.ins
    bt = q.dtype
    o_seq, dq_seq, dk_seq, dv_seq = layer.outs
    oh, dqh, dkh, dvh, lse = layer.oh, layer.dqh, layer.dkh, layer.dvh, layer.lse
    ws_f, ws_b = layer.ws_f, layer.ws_b
    stream = layer.stream
    full = layer.full
    outs_main = layer.outs
    step = layer.step

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def check(where):
        st, site = uly.ulysses_get_device_status()
        if st != 0:
            raise RuntimeError(f"device status {st} at site {site:#x} {where}")

    # ---- timed region: device time, inputs resident in HBM
    with ClockSampler(dev.index, args.clock_log_dir) as clk:
        elapsed_ms, ph = layer.time(args.steps, args.warmup, barrier, check)
    elapsed_ms = max_over_ranks(elapsed_ms, dist, dev)

    # ---- the same step through the fused seq-layout calls (no swaps)
    fused = None
    if full and (N // P) % 128 == 0:
        def fused_step():
            uly.ulysses_attn_fwd_seq(q, k, v, o_seq, lse, P, causal=w.causal, cu_seqlens=cu, workspace=ws_f)
            uly.ulysses_attn_bwd_seq(q, k, v, o_seq, lse, do, dq_seq, dk_seq, dv_seq, P, causal=w.causal,
                                     cu_seqlens=cu, workspace=ws_b)
        for _ in range(2):
            fused_step()
        barrier()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(args.steps):
            fused_step()
        f1.record(stream)
        barrier()
        fused_ms = max_over_ranks(f0.elapsed_time(f1) / args.steps, dist, dev)
        fused = {"ms_per_step": fused_ms, "launches_per_step": 1 + 3}
        st, site = uly.ulysses_get_device_status()
        if st != 0:
            raise RuntimeError(f"device status {st} at site {site:#x} in the fused timing")

    # ---- ring attention on the same inputs (chunks of the seq layout, all heads)
    ring = None
    ring_skipped = None
    if w.packed_docs and full and not args.no_ring:
        # the ring path computes plain causal / non-causal attention: timing it on
        # this workload would time a different (larger) computation
        ring_skipped = "ring attention takes no document mask; not timed on a packed-document workload"
    if full and not args.no_ring and not w.packed_docs:
        Np = N // P
        lse_r = torch.empty(P, B, w.Hq, Np, dtype=torch.float32, device=dev)
        ws_rf = torch.empty(uly.load().ulysses_ring_attn_workspace_size(B, N, w.Hq, w.Hkv, d, P, 0,
                                                                       0 if bt == torch.bfloat16 else 1),
                            dtype=torch.uint8, device=dev)
        ws_rb = torch.empty(uly.load().ulysses_ring_attn_workspace_size(B, N, w.Hq, w.Hkv, d, P, 1,
                                                                       0 if bt == torch.bfloat16 else 1),
                            dtype=torch.uint8, device=dev)

        def ring_step():
            uly.ulysses_ring_attn_fwd(q, k, v, o_seq, lse_r, P, causal=w.causal, workspace=ws_rf)
            uly.ulysses_ring_attn_bwd(q, k, v, o_seq, lse_r, do, dq_seq, dk_seq, dv_seq, P, causal=w.causal,
                                      workspace=ws_rb)
        for _ in range(2):
            ring_step()
        barrier()
        r0 = torch.cuda.Event(enable_timing=True)
        r1 = torch.cuda.Event(enable_timing=True)
        r0.record(stream)
        for _ in range(args.steps):
            ring_step()
        r1.record(stream)
        barrier()
        ring_ms = max_over_ranks(r0.elapsed_time(r1) / args.steps, dist, dev)
        st, site = uly.ulysses_get_device_status()
        if st != 0:
            raise RuntimeError(f"device status {st} at site {site:#x} in the ring timing")
        es = 2 if bt == torch.bfloat16 else 4
        ring = {"ms_per_step": ring_ms}
        # per GPU and layer, forward + backward, if the P ranks were P GPUs:
        #   Ulysses: the four all-to-alls move (P-1)/P of the local Q,K,V,O and dO,dQ,dK,dV
        #   ring:    P-1 hops of the K,V chunk forward; K,V and the fp32 dK,dV accumulators backward
        ring["comm_model_bytes_per_gpu"] = {
            "ulysses": int((P - 1) / P * Np * B * 4 * (w.Hq + w.Hkv) * d * es),
            "ring": int((P - 1) * Np * B * 2 * w.Hkv * d * (es + es + 4))}
        del ws_rf, ws_rb, lse_r

    # ---- end to end: host buffers in pinned memory, copies inside the timed region.
    # Every step uploads its own Q, K, V, dO from pinned host memory and reads
    # its O, dQ, dK, dV back.  Served as a stream of batches: two sets of device
    # buffers, the upload of step i+1 (one copy stream) and the read-back of
    # step i-1 (another) run while step i computes; the timed region opens
    # before the first upload and closes after the last read-back.  A step
    # starts once its Q, K, V are in (dO is first read after the forward) and
    # its O is read back while its backward runs.  The same loop on one stream
    # (no overlap) is reported beside it.
    pin = lambda x: torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    h_in = [pin(x).copy_(x) for x in (q, k, v, do)]
    outs = outs_main if full else (oh, dqh, dkh, dvh)
    h_out = [[pin(x) for x in outs] for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in h_in)
    d2h = sum(x.numel() * x.element_size() for x in h_out[0])
    e_steps = max(2, args.steps)
    sets_in = [(q, k, v, do), tuple(torch.empty_like(x) for x in (q, k, v, do))]
    # a second output set only where the results are written in the seq layout
    sets_out = [outs_main, tuple(torch.empty_like(x) for x in outs_main) if full else outs_main]
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def result_of(i):  # the device tensors step i's read-back copies
        return sets_out[i % 2] if full else outs

    barrier()
    e0, e1 = pipelined_steps(e_steps, stream, up, down, step, sets_in, sets_out, result_of,
                             lambda i: h_in, lambda i: h_out[i % 2], one_output_set=not full)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, dist, dev)
    # the same work with no overlap: upload, step, read-back on one stream
    s0 = torch.cuda.Event(enable_timing=True)
    s1 = torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for i in range(e_steps):
        for dx, hx in zip(sets_in[0], h_in):
            dx.copy_(hx, non_blocking=True)
        step(ins=sets_in[0], outs_seq=sets_out[0])
        for hx, dx in zip(h_out[0], result_of(0)):
            hx.copy_(dx, non_blocking=True)
    s1.record(stream)
    barrier()
    e2e_serial_ms = max_over_ranks(s0.elapsed_time(s1) / e_steps, dist, dev)
    st, site = uly.ulysses_get_device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} at site {site:#x} in the end-to-end timing")
    del sets_in, sets_out

    # ---- the sequence-parallel loss on the same tokens (Qwen3 vocabulary)
    loss = None
    if not args.no_loss and full:
        V = args.vocab
        del h_in, h_out
        torch.cuda.empty_cache()
        g = torch.Generator(device=dev)
        g.manual_seed(args.seed + 7)
        logits = torch.randn(P, B, N // P, V, device=dev, dtype=torch.bfloat16, generator=g)
        labels = torch.randint(0, V, (P, B, N // P), device=dev, generator=g)
        dlogits = torch.empty_like(logits)
        ws_l = torch.empty(uly.load().ulysses_sharded_ce_workspace_size(B, N, P), dtype=torch.uint8, device=dev)
        for _ in range(2):
            uly.ulysses_sharded_ce_loss(logits, labels, P, dlogits=dlogits, workspace=ws_l)
        barrier()
        l0 = torch.cuda.Event(enable_timing=True)
        l1 = torch.cuda.Event(enable_timing=True)
        l0.record(stream)
        n_rep = 3
        for _ in range(n_rep):
            uly.ulysses_sharded_ce_loss(logits, labels, P, dlogits=dlogits, workspace=ws_l)
        l1.record(stream)
        barrier()
        loss_ms = l0.elapsed_time(l1) / n_rep
        st, site = uly.ulysses_get_device_status()
        if st != 0:
            raise RuntimeError(f"device status {st} at site {site:#x} in the loss timing")
        alg = 2 * logits.numel() * logits.element_size()  # read the logits once, write the gradient once
        loss = {"what": "ulysses_sharded_ce_loss with the gradient: shifted labels, per-rank CE, "
                        "good-token-weighted aggregation, d loss / d logits",
                "tokens": B * N, "vocab": V, "dtype": "bf16", "ms": round(loss_ms, 3),
                "algorithmic_bytes": alg, "gbps": round(alg / (loss_ms * 1e-3) / 1e9, 1),
                "frac_of_hbm": round(alg / (loss_ms * 1e-3) / 1e9 / _peaks()[0], 3),
                "note": "with the gradient each row is held on chip by a cluster of 1, 2, 4 or 8 CTAs "
                        "(by vocabulary size; 4 for 151936 in bf16): one HBM read and one write per "
                        "logit, the algorithmic bytes"}
        del logits, labels, dlogits, ws_l
        torch.cuda.empty_cache()

    fwd_flops, bwd_flops = _flops(w, cu)
    step_flops = fwd_flops + bwd_flops
    ms = elapsed_ms / args.steps
    value = whole_job_throughput(world, step_flops, ms)
    hbm, tc_burst, tc_sus, src = _peaks()
    swap_bytes = layer.swap_bytes()
    # phases 0, 2 and 4 hold every swap (2 = O back to seq + dO to head)
    swap_ms = ph[0] + ph[2] + ph[4]
    bwd_tflops = bwd_flops / (ph[3] * 1e-3) / 1e12
    fwd_tflops = fwd_flops / (ph[1] * 1e-3) / 1e12
    traffic = None
    tr_path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if os.path.exists(tr_path):
        try:
            tr = json.load(open(tr_path)).get("attn_bwd_bf16_kernel")
            src_hash = hashlib.sha256(open(os.path.join(
                ROOT, "long_context_sequence_head_gb300", "csrc", "attn_bwd_bf16.cu"), "rb").read()).hexdigest()
            if tr and tr.get("src_sha256") == src_hash and tr.get("workload") == args.workload:
                traffic = tr.get("dram_bytes_per_launch")
        except Exception:
            traffic = None
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded N(0,1) Q/K/V/dO of the workload's shapes)",
        "config": _config(w, args, world),
        "tokens_per_s": round(world * B * N / (ms * 1e-3), 1),
        "attn_fwd_tflops": round(fwd_tflops, 1), "attn_bwd_tflops": round(bwd_tflops, 1),
        "attn_fwd_bwd_tflops": round(step_flops / ((ph[1] + ph[3]) * 1e-3) / 1e12, 1),
        "attn_fwd_bwd_frac_of_bf16_peak": round(step_flops / ((ph[1] + ph[3]) * 1e-3) / 1e12 / tc_sus, 3),
        "flops_no_recompute_tflops": round((fwd_flops * 3.0) / (ms * 1e-3) / 1e12, 2),
        "swap_gbps": round(swap_bytes / (swap_ms * 1e-3) / 1e9, 1),
        "swap_frac_of_hbm": round(swap_bytes / (swap_ms * 1e-3) / 1e9 / hbm, 3),
        "phase_ms": {"swap_qkv": round(ph[0], 3), "attn_fwd": round(ph[1], 3),
                     "swap_o_and_do": round(ph[2], 3), "attn_bwd": round(ph[3], 3),
                     "swap_dq_dk_dv": round(ph[4], 3)},
        "roofline": {"kernel": "ulysses_attn_bwd (bwd_pre + attn_bwd_bf16_kernel + dq_convert)",
                     "bound": "tensor", "achieved": round(bwd_tflops, 1), "peak": tc_sus, "unit": "TFLOP/s",
                     "frac": round(bwd_tflops / tc_sus, 3), "traffic": traffic,
                     "peak_source": f"{src} bf16 sustained (MEASURED_PEAKS.json)" if src == "measured"
                     else "fallback 1.7 PFLOP/s sustained"},
        "e2e": {"value": round(whole_job_throughput(world, step_flops, e2e_ms), 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
                "how": "pinned host buffers; per step an upload of the inputs and a read-back of the "
                       "results, overlapped with the neighbouring steps' compute on two copy streams; "
                       "a step starts once its Q, K, V are in and its O is read back during its backward",
                "steps": e_steps, "serial_ms_per_step": round(e2e_serial_ms, 3),
                "serial_value": round(whole_job_throughput(world, step_flops, e2e_serial_ms), 2)},
        "fused_seq_layout_path": None if fused is None else {
            "what": "ulysses_attn_fwd_seq + ulysses_attn_bwd_seq: same step without the swap kernels",
            "ms_per_step": round(fused["ms_per_step"], 3),
            "value": round(whole_job_throughput(world, step_flops, fused["ms_per_step"]), 2), "unit": UNIT,
            "tokens_per_s": round(world * B * N / (fused["ms_per_step"] * 1e-3), 1)},
        "ring_attention": ({"skipped": ring_skipped} if ring_skipped else None) if ring is None else {
            "what": "ulysses_ring_attn_fwd + ulysses_ring_attn_bwd on the same inputs: P chunks of all heads, "
                    "P ring steps merged through the log-sum-exp (one GPU: the hops are pointer offsets)",
            "ms_per_step": round(ring["ms_per_step"], 3),
            "value": round(whole_job_throughput(world, step_flops, ring["ms_per_step"]), 2), "unit": UNIT,
            "comm_model_bytes_per_gpu_per_layer": ring["comm_model_bytes_per_gpu"]},
        "sharded_loss": loss,
        "clocks": clk.summary(),
        "gpu_launches": args.steps * layer.launches_per_step,
    }
    return line


# ------------------------------------------------------------ oracle arm
def oracle_inputs(w, seed, want_dout=True, device="cpu"):
    """The workload's inputs in the oracle's head layout, upcast to fp64 once
    (outside any timed region).  device="cuda" draws them with the seeded
    generator on the GPU (the bytes the GPU arm times, and fast for the 1M
    workload) before they are copied to the host."""
    import oracle
    from ulysses_inputs import draw_seq_inputs
    seq = draw_seq_inputs(w, seed=seed, device=device, want_dout=want_dout)
    out = {}
    for n in list(seq):
        x = seq.pop(n).cpu()
        out[n] = oracle._f64(oracle.seq_to_head(x, w.P)[: w.shards_timed])
        del x
    return out


def oracle_workload_baseline(w, cu, seed):
    """The fp64 oracle, as it stands, on a bounded sample of one workload
    (a few seconds of host work): the whole forward and backward for the
    tiny workload, random query rows (forward + dQ) for the N=8192 and
    packed-document workloads, and 256 random forward rows (O, lse) of the
    one timed head shard for the 1M workload.  Credited FLOPs: the step's
    algorithmic FLOPs for the full case; 4*d per allowed pair for a forward
    row and 6*d for a dQ row."""
    import numpy as np
    import oracle
    heads = oracle_inputs(w, seed, want_dout=w.N < (1 << 20), device="cuda")
    rng = np.random.default_rng(seed)
    S = w.shards_timed

    def allowed(i):
        if cu is None:
            return i + 1
        kk = int(np.searchsorted(cu, i, side="right")) - 1
        return i - int(cu[kk]) + 1
    if w.N <= 1024:
        fwd, bwd = _flops(w, cu)
        reps = 0
        t0 = time.perf_counter()
        while reps == 0 or time.perf_counter() - t0 < 1.0:
            oracle.attn_bwd(heads["q"], heads["k"], heads["v"], heads["dout"], causal=w.causal, cu_seqlens=cu)
            reps += 1
        dt = time.perf_counter() - t0
        credit = reps * (fwd + bwd)
        sample = f"the whole forward and backward of {w.name} (all {S} head shards), {reps} times"
    elif w.N < (1 << 20):
        rows = [(int(rng.integers(S)), 0, int(rng.integers(w.Hp)), int(rng.integers(w.N))) for _ in range(8192)]
        credit = sum(10 * w.d * allowed(i) for *_, i in rows)
        t0 = time.perf_counter()
        oracle.attn_fwd_rows(heads["q"], heads["k"], heads["v"], rows, cu_seqlens=cu)
        oracle.attn_bwd_q_rows(heads["q"], heads["k"], heads["v"], heads["dout"], rows, cu_seqlens=cu)
        dt = time.perf_counter() - t0
        sample = f"8192 random query rows (forward + dQ) of {w.name}"
    else:
        rows = [(0, 0, int(rng.integers(w.Hp)), int(rng.integers(w.N))) for _ in range(256)]
        credit = sum(4 * w.d * allowed(i) for *_, i in rows)
        t0 = time.perf_counter()
        oracle.attn_fwd_rows(heads["q"], heads["k"], heads["v"], rows, cu_seqlens=cu)
        dt = time.perf_counter() - t0
        sample = f"256 random forward rows (O, lse) of the timed head shard of {w.name}"
    return {"value": credit / dt / 1e12, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": sample, "seconds": round(dt, 2)}


def run_other_workloads(args, with_cpu_baseline):
    """The configurations beside the headline one, each timed on the same
    step (swaps, forward, backward) with its own warm-up, and, on request,
    the oracle timed on a bounded sample of it."""
    import argparse as _ap
    import torch
    import long_context_sequence_head_gb300 as uly
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    hbm, _, tc_sus, _ = _peaks()

    def barrier():
        torch.cuda.synchronize()

    def check(where):
        st, site = uly.ulysses_get_device_status()
        if st != 0:
            raise RuntimeError(f"device status {st} at site {site:#x} {where}")
    out = {}
    for name, steps, warmup in OTHER_WORKLOADS:
        w, cu = _workload(name)
        torch.cuda.empty_cache()
        layer = Layer(uly, w, cu, dev, args.seed)
        total_ms, ph = layer.time(steps, warmup, barrier, check)
        r = _rates(w, cu, layer, total_ms / steps, ph, tc_sus, hbm)
        r.update({"steps": steps, "warmup": warmup, "dtype": w.dtype,
                  "config": _config(w, _ap.Namespace(workload=name, seq_len=None), 1),
                  "gpu_launches": steps * layer.launches_per_step})
        del layer
        torch.cuda.empty_cache()
        if with_cpu_baseline:
            r["cpu_baseline"] = oracle_workload_baseline(w, cu, args.seed)
        out[name] = r
    return out


def oracle_sample(w, cu, heads, rows_per_step, seed):
    """Time the fp64 oracle on sampled query rows of the workload: forward
    rows (O, lse) and dQ rows.  Credited FLOPs: 4*d per allowed pair for a
    forward row (two products), 6*d per allowed pair for a dQ row (scores,
    dP and dQ products).  Returns (credited_flops, seconds, sample_text)."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(seed)
    S = w.shards_timed
    rows = [(int(rng.integers(S)), 0, int(rng.integers(w.Hp)), int(rng.integers(w.N)))
            for _ in range(rows_per_step)]

    def allowed(i):
        if cu is None:
            return i + 1
        k = int(np.searchsorted(cu, i, side="right")) - 1
        return i - int(cu[k]) + 1
    credit = sum(10 * w.d * allowed(i) for *_, i in rows)
    t0 = time.perf_counter()
    oracle.attn_fwd_rows(heads["q"], heads["k"], heads["v"], rows, cu_seqlens=cu)
    oracle.attn_bwd_q_rows(heads["q"], heads["k"], heads["v"], heads["dout"], rows, cu_seqlens=cu)
    dt = time.perf_counter() - t0
    return credit, dt, f"{rows_per_step} random query rows (forward + dQ) of {w.name}"


def run_reference(args, rank, world):
    import oracle
    w, cu = _workload(args.workload, args.seq_len)
    oracle.build()
    cores = oracle.num_threads()
    heads = oracle_inputs(w, args.seed)
    rows = args.oracle_rows
    for i in range(args.warmup):
        oracle_sample(w, cu, heads, max(1, rows // 8), args.seed + 1000 + i)
    tot_c, tot_t = 0.0, 0.0
    sample = ""
    for i in range(args.steps):
        c, t, sample = oracle_sample(w, cu, heads, rows, args.seed + 1 + i)
        tot_c += c
        tot_t += t
    value = tot_c / tot_t / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot_t / args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) Q/K/V/dO of the workload's shapes)", "config": _config(w, args, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"per step: {sample}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen3_4b_n65536")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--seq-len", type=int, default=None,
                    help="override the workload's N (profiling smaller cases of the same kernels)")
    ap.add_argument("--oracle-rows", type=int, default=8192)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clock-log-dir", default="",
                    help="directory for the raw nvidia-smi clock samples (default: the system temp dir)")
    ap.add_argument("--no-loss", action="store_true", help="skip the sequence-parallel loss measurement")
    ap.add_argument("--no-ring", action="store_true", help="skip the ring-attention measurement")
    ap.add_argument("--vocab", type=int, default=151936, help="vocabulary of the loss measurement (Qwen3)")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="time only the headline workload (skip the N=8192, packed, tiny and 1M lines)")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return

    dist = None
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    line = run_ours(args, rank, world, dist)
    if world == 1 and not args.no_other_workloads and args.seq_len is None:
        line["other_workloads"] = run_other_workloads(args, with_cpu_baseline=not args.no_cpu_baseline)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        w, cu = _workload(args.workload, args.seq_len)
        import oracle
        oracle.build()
        heads = oracle_inputs(w, args.seed)
        c, t, sample = oracle_sample(w, cu, heads, args.oracle_rows, args.seed + 100)
        line["cpu_baseline"] = {"value": c / t / 1e12, "unit": UNIT, "cores": oracle.num_threads(),
                                "kind": "oracle", "sample": sample, "seconds": round(t, 2)}
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
