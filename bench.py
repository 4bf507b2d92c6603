#!/usr/bin/env python3
"""Benchmark of the gated DeltaNet token mixer on one GB300 (or N replicas).

A step is one pass of the whole hot path over one batch of synthetic input:
  * prefill: one sequence of T=8192 tokens, H_k=16 tiled to H_v=48, bf16
    activations, zero initial state (gdn_prefill_chunked, chunk = 64);
  * decode: B=64 sequences, one token each, H_k=16 / H_v=32, bf16, fp32 state
    updated in place (gdn_decode_step);
  * speculative verify: the same B=64 sequences, K=3 tokens each, with
    per-position checkpoints on a state ring (gdn_verify_k_ring), then
    gdn_commit_ring of a seeded accept length in {1,2,3} (the accepted
    checkpoint becomes the live state where it lies; only conv rows move).
value = tokens processed per second over the step (8192 + 64 + 192 tokens);
the per-part figures (tokens/s, ms, roofline) are under "parts".

Timing: CUDA events on the launching stream, W >= 3 warm-up steps, L2 flushed
(a 256 MiB write) before every timed step, outside the timed region; every
input is also larger than L2.  e2e: the same step through the C ABI with the
step's inputs copied from pinned host memory and its outputs read back, inside
the timed region, the copies pipelined against the compute on two side streams:
the decode and verify inputs first (those calls run while the prefill's inputs
arrive), then the prefill's 8192 tokens through gdn_prefill_chunked in 4
segments of 2048 (state carried on the device; the chunk grid, hence every
result, is that of one call), segment i+1's inputs copied in while segment i
runs and each segment's outputs copied out as soon as it is done.  Under torchrun (N > 1) each rank runs its own replica (no
collective on the data path: the layer shards by sequence and head) and the
slowest rank's time is used.

"extras" (skipped with --no-extras) times the two other configurations outside
the step: decode at batch 1 as 1000 in-place steps captured in one CUDA graph,
and the packed varlen prefill (8 sequences, T=65536, nonzero initial state).

--impl reference times the CPU oracle (fp64, OpenMP) on the host cores over
whole steps of the same workload (about a second each), nothing extrapolated.
"""
from __future__ import annotations

import argparse
import json
import math
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

import gdn_inputs  # noqa: E402

METRIC = "GDN layer tokens/s: prefill T=8192 & decode B=64; % of roofline"
WORKLOAD = ("prefill T=8192 H_k=16 H_v=48 bf16 (chunk 64) + decode B=64 H_k=16 H_v=32 bf16 "
            "+ verify B=64 K=3 + commit (state ring)")
L2_FLUSH_BYTES = 256 << 20
TOKENS_PER_STEP = 8192 + 64 + 64 * 3   # prefill T + decode B + verify B * K


# ------------------------------------------------------------------ algorithmic work
def prefill_bytes(T, Hk, Hv, out_bytes=2, act_bytes=2, init_state=False, n_seq=1):
    C = 128 * (2 * Hk + Hv)
    HvD = Hv * 128
    b = T * C * act_bytes + T * HvD * act_bytes + 2 * T * Hv * act_bytes + T * HvD * out_bytes
    b += n_seq * (Hv * 128 * 128 * 4 + 3 * C * act_bytes)       # final S and conv state written
    if init_state:
        b += n_seq * (Hv * 128 * 128 * 4 + 3 * C * act_bytes)   # initial state read
    b += C * 16 + Hv * 8 + 128 * 4                              # weights
    return b


def decode_bytes(B, Hk, Hv, K=1, act_bytes=2, out_bytes=2, ckpt=False, state_bytes=4):
    C = 128 * (2 * Hk + Hv)
    per_seq = 2 * Hv * 128 * 128 * state_bytes if not ckpt else Hv * 128 * 128 * state_bytes * (1 + K)
    per_seq += (3 * C * act_bytes) * (2 if not ckpt else 1 + K)
    per_seq += K * (C + Hv * 128 + 2 * Hv) * act_bytes + K * Hv * 128 * out_bytes
    return B * per_seq + C * 16 + Hv * 8 + 128 * 4


def prefill_flops(T, Hv):
    # chunk-64 form, triangles counted once: 1.41e5 flop per token per v-head
    C_, d = 64, 128
    per = (C_ * (C_ - 1) * d / C_ + C_ * C_ / 3 + 2 * (C_ + 1) * d + 2 * d * d + (C_ + 1) * d
           + 2 * d * d + (C_ + 1) * d + 2 * d * d + 2 * d)
    return per * T * Hv


# The sources that decide each part's kernels, launch shapes and memory traffic.
_COMMON_SOURCES = ("gdn_api.cu", "gdn_common.cuh", "gdn_internal.h", "gdn_tc.cuh")
PART_SOURCES = {
    "prefill": _COMMON_SOURCES + ("gdn_prefill_tc.cu", "gdn_prefill_prep.cuh", "gdn_prefill_chain.cuh",
                                  "gdn_prefill_simt.cu", "gdn_prefill_tc.cuh", "gdn_tma.cu"),
    "decode": _COMMON_SOURCES + ("gdn_recurrent.cu", "gdn_recurrent_stream.cu"),
}


def kernel_sources_hash(part: str) -> str:
    """sha256 over the sources of one part (PART_SOURCES, in that order) and the public header."""
    import hashlib
    csrc = os.path.join(ROOT, "gated_deltanet_linear_decode_gb300", "csrc")
    files = [os.path.join(csrc, f) for f in PART_SOURCES[part]] + [os.path.join(ROOT, "include", "gdn.h")]
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic() -> dict:
    """DRAM bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum) recorded in
    profiles/traffic.json, for each part whose sources are unchanged since they were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return {}
    return {k: v["bytes"] for k, v in rec.get("parts", {}).items()
            if k in PART_SOURCES and v.get("sources_sha256") == kernel_sources_hash(k)}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.proc = None
        self.lines = []
        self.bus = None
        try:
            pr = torch.cuda.get_device_properties(device_index)
            if hasattr(pr, "pci_bus_id"):
                self.bus = f"{getattr(pr, 'pci_domain_id', 0):08X}:{pr.pci_bus_id:02X}:{getattr(pr, 'pci_device_id', 0):02X}.0"
        except Exception:
            pass

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.bus:
            cmd.insert(1, f"--id={self.bus}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "samples": len(sm),
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons)}


# ------------------------------------------------------------------ the GPU arm
class Workload:
    """Device-resident inputs/outputs of one step, plus pinned host copies for e2e."""

    @staticmethod
    def _packed(named, dev):
        """One pinned host buffer and one device buffer holding the tensors of `named` (a list of
        (dict, key, tensor)), each at a 256-byte aligned offset, so that all of them move in one
        copy; returns (host buffer, device buffer, [(dict, key, host view, device view)])."""
        off, place = 0, []
        for d, k, t in named:
            nb = t.numel() * t.element_size()
            place.append((d, k, t, off, nb))
            off = (off + nb + 255) // 256 * 256
        hbuf = torch.empty(off, dtype=torch.uint8).pin_memory()
        dbuf = torch.empty(off, dtype=torch.uint8, device=dev)
        views = []
        for d, k, t, o, nb in place:
            hv = hbuf[o:o + nb].view(t.dtype).view(t.shape)
            hv.copy_(t)
            views.append((d, k, hv, dbuf[o:o + nb].view(t.dtype).view(t.shape)))
        return hbuf, dbuf, views

    def __init__(self, device, prefill_tokens=8192):
        import gated_deltanet_linear_decode_gb300 as gdn
        self.gdn = gdn
        dev = device
        # the prefill workload (a shorter sequence of the same shape only for profiling runs)
        self.pc = (gdn_inputs.prefill_t8192() if prefill_tokens == 8192 else
                   gdn_inputs.make_case(f"prefill T={prefill_tokens} Hk=16 Hv=48 bf16", Hk=16, Hv=48,
                                        lengths=[prefill_tokens], S0="zero", conv0="zero", seed=1002))
        self.dc = gdn_inputs.decode_b64()
        self.vc = gdn_inputs.verify_b64_k3()
        pc, dc, vc = self.pc, self.dc, self.vc
        self.p_dims = gdn.make_dims(pc.Hk, pc.Hv, torch.bfloat16, torch.bfloat16)
        self.d_dims = gdn.make_dims(dc.Hk, dc.Hv, torch.bfloat16, torch.bfloat16)
        self.p_w = gdn.make_weights(pc.conv_w, pc.dt_bias, pc.ssm_a, pc.norm_w, device=dev)
        self.d_w = gdn.make_weights(dc.conv_w, dc.dt_bias, dc.ssm_a, dc.norm_w, device=dev)
        # host (pinned) inputs for the e2e leg
        pin = lambda t: t.contiguous().pin_memory()
        self.h = {k: pin(getattr(pc, k)) for k in ("x", "z", "a_raw", "b_raw")}
        # the decode and verify inputs (a few MB in eight tensors) packed in one pinned buffer and
        # one device buffer, so that the e2e leg moves them in one copy
        self.hd, self.hv, self.d_in, self.v_in = {}, {}, {}, {}
        self.h_small, self.d_small, views = self._packed(
            [(0, k, getattr(dc, k).contiguous()) for k in ("x", "z", "a_raw", "b_raw")] +
            [(1, k, getattr(vc, k).contiguous()) for k in ("x", "z", "a_raw", "b_raw")], dev)
        for which, k, hview, dview in views:
            (self.hd if which == 0 else self.hv)[k] = hview
            (self.d_in if which == 0 else self.v_in)[k] = dview
        self.d_small.copy_(self.h_small)
        # device copies of the prefill inputs
        self.p_in = {k: v.to(dev, non_blocking=True) for k, v in self.h.items()}
        self.cu_h = pc.cu_seqlens.to(torch.int32)
        self.cu_d = self.cu_h.to(dev)
        self.p_conv = torch.zeros(1, 3, pc.C, device=dev, dtype=torch.bfloat16)
        self.p_S = torch.zeros(1, pc.Hv, 128, 128, device=dev)
        self.p_out = torch.empty(pc.T, pc.Hv * 128, device=dev, dtype=torch.bfloat16)
        nws = gdn.gdn_prefill_workspace_bytes(self.p_dims, 1, pc.T)
        self.p_ws = torch.empty(max(nws, 16), device=dev, dtype=torch.uint8) if nws else None
        self.d_conv = dc.conv0.to(dev)
        self.d_S = dc.S0.to(dev)
        # decode and verify outputs: one device buffer and one pinned host buffer (one copy out)
        n_d, n_v = dc.N * dc.Hv * 128, vc.N * vc.K * vc.Hv * 128
        self.d_small_out = torch.empty(n_d + n_v, device=dev, dtype=torch.bfloat16)
        self.h_small_out = torch.empty(n_d + n_v, dtype=torch.bfloat16).pin_memory()
        self.d_out = self.d_small_out[:n_d].view(dc.N, dc.Hv * 128)
        B, K = vc.N, vc.K
        self.v_ckc = torch.empty(B, K, 3, vc.C, device=dev, dtype=torch.bfloat16)
        self.v_ckS = torch.empty(B, K, vc.Hv, 128, 128, device=dev)
        self.v_out = self.d_small_out[n_d:].view(B * K, vc.Hv * 128)
        self.acc = vc.accept_len.to(dev)
        # the same verify + commit on a state ring (R = K + 1 slots, slot 0 live at the start)
        self.r_S = torch.zeros(B, K + 1, vc.Hv, 128, 128, device=dev)
        self.r_S[:, 0] = vc.S0.to(dev)
        self.r_cur = torch.zeros(B, device=dev, dtype=torch.int32)
        self.r_conv = vc.conv0.to(dev)
        self.h_pout = torch.empty(self.p_out.shape, dtype=torch.bfloat16).pin_memory()
        self.h_dout = self.h_small_out[:n_d].view(self.d_out.shape)
        self.h_vout = self.h_small_out[n_d:].view(self.v_out.shape)
        self.flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev, dtype=torch.float32)
        self.launches_per_step = 0

    # each call returns the number of library kernels it launched
    def prefill(self):
        g, i = self.gdn, self.p_in
        g.gdn_prefill_chunked(self.p_dims, self.p_w, self.cu_h, self.cu_d, i["x"], i["z"], i["a_raw"], i["b_raw"],
                              self.p_conv, self.p_S, self.p_out, zero_init=True, workspace=self.p_ws)
        # chunk table, the prefill kernel (preparation and chain roles side by side), conv-state update
        return 3

    def decode(self):
        g, i = self.gdn, self.d_in
        g.gdn_decode_step(self.d_dims, self.d_w, i["x"], i["z"], i["a_raw"], i["b_raw"], self.d_conv, self.d_S,
                          self.d_out)
        return 1

    def verify_copy(self):
        """Verify + commit on plain states (the accepted checkpoint is copied back)."""
        g, i = self.gdn, self.v_in
        g.gdn_verify_k(self.d_dims, self.d_w, self.vc.K, i["x"], i["z"], i["a_raw"], i["b_raw"], self.d_conv,
                       self.d_S, self.v_ckc, self.v_ckS, self.v_out)
        g.gdn_commit(self.d_dims, self.vc.K, self.acc, self.v_ckc, self.v_ckS, self.d_conv, self.d_S)
        return 2

    def verify_only(self):
        g, i = self.gdn, self.v_in
        g.gdn_verify_k(self.d_dims, self.d_w, self.vc.K, i["x"], i["z"], i["a_raw"], i["b_raw"], self.d_conv,
                       self.d_S, self.v_ckc, self.v_ckS, self.v_out)
        return 1

    def verify(self):
        """The step's verify: verify walk + commit on the state ring (the commit moves no state)."""
        return self.verify_ring()

    def verify_ring(self):
        g, i = self.gdn, self.v_in
        g.gdn_verify_k_ring(self.d_dims, self.d_w, self.vc.K, i["x"], i["z"], i["a_raw"], i["b_raw"], self.r_conv,
                            self.r_S, self.r_cur, self.v_ckc, self.v_out)
        g.gdn_commit_ring(self.d_dims, self.vc.K, self.vc.K + 1, self.acc, self.v_ckc, self.r_conv, self.r_cur)
        return 2

    @staticmethod
    def e2e_segments(T):
        """Prefill segments of the e2e step: 2048 tokens each, the last 2048 cut into 1024 + 768 +
        256 (T = 8192: 2048, 2048, 2048, 1024, 768, 256 -- the fastest of the splits measured:
        short last segments leave little compute and copying once the last inputs land, while
        every call costs a fixed ~60 us of start-up); one segment when T is not a multiple of 64."""
        if T % 64 or T < 1024:
            return (T,)
        segs = [2048] * (T // 2048) + ([T % 2048] if T % 2048 else [])
        last = segs.pop()
        if last == 2048:
            tail = [1024, 768, 256]
        elif last >= 512:
            tail = [last - 256, 256]
        else:
            tail = [last]
        return tuple(segs + tail)

    def e2e_step(self, segs=None):
        """One step from host buffers to host buffers through the C ABI, with the transfers
        pipelined against the compute on two side streams.  The decode and verify inputs (a few
        MB) go first, so those two calls run while the prefill's inputs are still arriving; the
        prefill's tokens then go through gdn_prefill_chunked in segments of `segs` tokens
        (multiples of 64: the conv and recurrent state carried on the device from one call to
        the next, the chunk grid unchanged, so the results are those of one call), segment i+1's
        inputs copied in while segment i computes and each segment's outputs copied out as soon
        as it is done.  The host enqueues the copies one segment ahead of the compute (so the
        copy engine never waits for the host, and no launch waits behind the host issuing all
        the copies); the last segments are short, so little compute and copying is left once
        the last inputs land.
        Returns the number of library kernels launched."""
        cur = torch.cuda.current_stream()
        if not hasattr(self, "s_in"):
            self.s_in, self.s_out = torch.cuda.Stream(self.p_out.device), torch.cuda.Stream(self.p_out.device)
        segs = self.e2e_segments(self.pc.T) if segs is None else tuple(segs)
        assert sum(segs) == self.pc.T and (len(segs) == 1 or all(L > 0 and L % 64 == 0 for L in segs))
        if not hasattr(self, "cu_seg"):
            self.cu_seg = {}
        for L in segs:
            if L not in self.cu_seg:   # one segment table per length, made outside the timed steps
                h = torch.tensor([0, L], dtype=torch.int32)
                self.cu_seg[L] = (h, h.to(self.p_out.device))
        self.s_in.wait_stream(cur)
        self.s_out.wait_stream(cur)
        starts = [sum(segs[:i]) for i in range(len(segs))]
        pi = self.p_in
        ev_in = [torch.cuda.Event() for _ in segs]

        def copy_in(i):   # segment i's inputs, on the input stream
            sl = slice(starts[i], starts[i] + segs[i])
            with torch.cuda.stream(self.s_in):
                for k in self.h:
                    pi[k][sl].copy_(self.h[k][sl], non_blocking=True)
                ev_in[i].record(self.s_in)

        ev_small, ev_dv = torch.cuda.Event(), torch.cuda.Event()
        with torch.cuda.stream(self.s_in):
            self.d_small.copy_(self.h_small, non_blocking=True)   # the decode and verify inputs
            ev_small.record(self.s_in)
        copy_in(0)   # the copy engine keeps one segment queued ahead of the compute
        cur.wait_event(ev_small)
        n = self.decode() + self.verify()
        ev_dv.record(cur)
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(ev_dv)
            self.h_small_out.copy_(self.d_small_out, non_blocking=True)   # the decode and verify outputs
        for i, L in enumerate(segs):
            if i + 1 < len(segs):
                copy_in(i + 1)
            sl = slice(starts[i], starts[i] + L)
            cur.wait_event(ev_in[i])
            cu_h, cu_d = self.cu_seg[L]
            self.gdn.gdn_prefill_chunked(self.p_dims, self.p_w, cu_h, cu_d, pi["x"][sl], pi["z"][sl],
                                         pi["a_raw"][sl], pi["b_raw"][sl], self.p_conv, self.p_S, self.p_out[sl],
                                         zero_init=(i == 0), workspace=self.p_ws)
            n += 3
            ev_done = torch.cuda.Event()
            ev_done.record(cur)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(ev_done)
                self.h_pout[sl].copy_(self.p_out[sl], non_blocking=True)
        cur.wait_stream(self.s_out)
        cur.wait_stream(self.s_in)
        return n

    def io_bytes(self):
        h2d = sum(t.numel() * t.element_size() for t in self.h.values()) + self.h_small.numel()
        d2h = sum(t.numel() * t.element_size() for t in (self.h_pout, self.h_small_out))
        return h2d, d2h

    def flush_l2(self):
        self.flush.fill_(1.0)


def run_gpu(args, rank, world):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    import gated_deltanet_linear_decode_gb300 as gdn
    gdn.library()
    wl = Workload(dev)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        wl.flush_l2()
        wl.prefill(); wl.decode(); wl.verify()
    torch.cuda.synchronize()

    parts = {"prefill": [], "decode": [], "verify": []}
    launches = 0
    sampler = ClockSampler(dev.index)
    sampler.start()
    _barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    step_ms = []
    for _ in range(args.steps):
        wl.flush_l2()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        ev[0].record(stream)
        launches += wl.prefill()
        ev[1].record(stream)
        launches += wl.decode()
        ev[2].record(stream)
        launches += wl.verify()
        ev[3].record(stream)
        torch.cuda.synchronize()
        parts["prefill"].append(ev[0].elapsed_time(ev[1]))
        parts["decode"].append(ev[1].elapsed_time(ev[2]))
        parts["verify"].append(ev[2].elapsed_time(ev[3]))
        step_ms.append(ev[0].elapsed_time(ev[3]))
    torch.cuda.synchronize()
    _barrier(world)
    wall = time.perf_counter() - t_wall0
    clocks = sampler.stop()

    # e2e: host buffers in, results out, inside the timed region (after W untimed steps that
    # create the side streams and the segment tables)
    for _ in range(args.warmup):
        wl.flush_l2()
        wl.e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for _ in range(max(1, args.steps)):
        wl.flush_l2()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        wl.e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))

    # outside the step: the verify walk alone, and verify + commit on plain states (the commit copies the
    # accepted checkpoint back)
    def timed_alone(fn):
        ms = []
        for it in range(args.warmup + max(1, args.steps)):
            wl.flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            if it >= args.warmup:
                ms.append(e0.elapsed_time(e1))
        return statistics.mean(ms)
    only_ms = timed_alone(wl.verify_only)
    copy_ms = timed_alone(wl.verify_copy)

    tot_ms = sum(step_ms)
    tot_ms = _max_over_ranks(tot_ms, world)
    e2e_tot = _max_over_ranks(sum(e2e_ms), world)
    pc, dc, vc = wl.pc, wl.dc, wl.vc
    tok_step = pc.T + dc.N + vc.N * vc.K
    assert tok_step == TOKENS_PER_STEP
    value = world * tok_step * args.steps / (tot_ms / 1e3)
    hbm, tf, peak_src = peaks()
    pm = statistics.mean(parts["prefill"])
    dm = statistics.mean(parts["decode"])
    vm = statistics.mean(parts["verify"])
    pb = prefill_bytes(pc.T, pc.Hk, pc.Hv)
    db = decode_bytes(dc.N, dc.Hk, dc.Hv)
    vb = decode_bytes(vc.N, vc.Hk, vc.Hv, K=vc.K, ckpt=True)
    pf = prefill_flops(pc.T, pc.Hv)
    traffic = measured_traffic()
    p_roof = {"bound": "hbm", "achieved": pb / (pm / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
              "frac": pb / (pm / 1e3) / 1e9 / hbm, "traffic": traffic.get("prefill"), "algorithmic_bytes": pb,
              "tensor_tflops_algorithmic": pf / (pm / 1e3) / 1e12, "peak_source": peak_src}
    d_roof = {"bound": "hbm", "achieved": db / (dm / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
              "frac": db / (dm / 1e3) / 1e9 / hbm, "traffic": traffic.get("decode"), "algorithmic_bytes": db,
              "peak_source": peak_src}
    v_roof = {"bound": "hbm", "achieved": vb / (vm / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
              "frac": vb / (vm / 1e3) / 1e9 / hbm, "traffic": None, "algorithmic_bytes": vb,
              "note": "verify walk + commit on the state ring (conv rows and slot index only)"}
    o_roof = {"bound": "hbm", "achieved": vb / (only_ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
              "frac": vb / (only_ms / 1e3) / 1e9 / hbm, "traffic": None, "algorithmic_bytes": vb,
              "note": "verify walk alone, timed outside the step"}
    c_roof = {"bound": "hbm", "achieved": vb / (copy_ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
              "frac": vb / (copy_ms / 1e3) / 1e9 / hbm, "traffic": None, "algorithmic_bytes_verify_only": vb,
              "note": "verify + commit on plain states (the commit copies the accepted checkpoint); "
                      "timed outside the step"}
    dominant = max((pm, "prefill", p_roof), (dm, "decode", d_roof), (vm, "verify", v_roof))[1:]
    h2d, d2h = wl.io_bytes()
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": tot_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 (bf16 activations in/out, fp32 state)",
        "data": "synthetic (seeded; no weights or dataset)",
        "config": step_config(world),
        "roofline": {**dominant[1], "kernel": dominant[0]},
        "parts": {
            "prefill_T8192": {"tokens_per_s": pc.T / (pm / 1e3), "ms": pm, "roofline": p_roof},
            "decode_B64": {"tokens_per_s": dc.N / (dm / 1e3), "ms": dm, "roofline": d_roof},
            "verify_B64_K3_commit_ring": {"tokens_per_s": vc.N * vc.K / (vm / 1e3), "ms": vm, "roofline": v_roof},
            "verify_B64_K3_alone": {"tokens_per_s": vc.N * vc.K / (only_ms / 1e3), "ms": only_ms, "roofline": o_roof},
            "verify_B64_K3_commit_copy": {"tokens_per_s": vc.N * vc.K / (copy_ms / 1e3), "ms": copy_ms,
                                          "roofline": c_roof},
        },
        "e2e": {"value": world * tok_step * len(e2e_ms) / (e2e_tot / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clocks,
        "wall_s_timed": wall,
    }
    return line


def run_extras(dev, warmup, reps):
    """The two other timed configurations, outside the step: decode at batch 1
    (1000 in-place steps captured in one CUDA graph; the 4.5 MB working set
    stays in L2, so its bandwidth is not an HBM figure) and the packed varlen
    prefill (8 sequences, T=65536, nonzero initial state, L2 flushed); the
    B=64 decode with a bf16 state; and the projections either side of the
    mixer at the prefill and decode sizes (L2 flushed)."""
    import gated_deltanet_linear_decode_gb300 as gdn
    hbm, tf, _ = peaks()
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, device=dev, dtype=torch.float32)
    out = {}

    def timed(fn, flush_l2):
        ms = []
        for it in range(warmup + reps):
            if flush_l2:
                flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            if it >= warmup:
                ms.append(e0.elapsed_time(e1))
        return statistics.mean(ms)

    def timed_graph(fn):
        """fn captured once in a CUDA graph, its replays timed: device time without the host's
        launch overhead (which is longer than these calls' device work)."""
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(2):
                fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            fn()
        torch.cuda.synchronize()
        return timed(g.replay, True)

    # decode B=1, 1000 steps per graph replay
    c = gdn_inputs.decode_b1()
    d = gdn.make_dims(c.Hk, c.Hv, torch.bfloat16, torch.bfloat16)
    w = gdn.make_weights(c.conv_w, c.dt_bias, c.ssm_a, c.norm_w, device=dev)
    i = {k: getattr(c, k).to(dev) for k in ("x", "z", "a_raw", "b_raw")}
    conv, S = c.conv0.to(dev), c.S0.to(dev)
    o = torch.empty(1, c.Hv * 128, device=dev, dtype=torch.bfloat16)
    n_steps = 1000
    step = lambda: gdn.gdn_decode_step(d, w, i["x"], i["z"], i["a_raw"], i["b_raw"], conv, S, o)
    side = torch.cuda.Stream(dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _ in range(3):
            step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for _ in range(n_steps):
            step()
    torch.cuda.synchronize()
    gm = timed(graph.replay, False)
    b1 = decode_bytes(1, c.Hk, c.Hv)
    out["decode_B1_graph_1000"] = {"tokens_per_s": n_steps / (gm / 1e3), "us_per_step": 1e3 * gm / n_steps,
                                   "launches_per_replay": n_steps, "bytes_per_step": b1,
                                   "achieved_GBps": b1 * n_steps / (gm / 1e3) / 1e9,
                                   "note": "state resident in L2 across steps; not an HBM roofline"}
    del graph

    # decode B=64 with the state stored as bf16 (same inputs as the step's decode)
    c = gdn_inputs.decode_b64()
    d = gdn.make_dims(c.Hk, c.Hv, torch.bfloat16, torch.bfloat16, state_dtype=torch.bfloat16)
    w = gdn.make_weights(c.conv_w, c.dt_bias, c.ssm_a, c.norm_w, device=dev)
    i = {k: getattr(c, k).to(dev) for k in ("x", "z", "a_raw", "b_raw")}
    conv, S = c.conv0.to(dev), c.S0.to(dev).to(torch.bfloat16)
    o = torch.empty(c.N, c.Hv * 128, device=dev, dtype=torch.bfloat16)
    bm = timed_graph(lambda: gdn.gdn_decode_step(d, w, i["x"], i["z"], i["a_raw"], i["b_raw"], conv, S, o))
    bb = decode_bytes(c.N, c.Hk, c.Hv, state_bytes=2)
    out["decode_B64_state_bf16"] = {"tokens_per_s": c.N / (bm / 1e3), "us": 1e3 * bm,
                                    "roofline": {"bound": "hbm", "achieved": bb / (bm / 1e3) / 1e9, "peak": hbm,
                                                 "unit": "GB/s", "frac": bb / (bm / 1e3) / 1e9 / hbm,
                                                 "algorithmic_bytes": bb}}
    del S, conv

    # decode B=64 with ssm_alpha / ssm_beta folded into the kernel (hidden 2048 -> a_raw, b_raw)
    c = gdn_inputs.decode_b64()
    pc = gdn_inputs.make_proj_case(T=c.N, H=2048, Hk=c.Hk, Hv=c.Hv, seed=11)
    d = gdn.make_dims(c.Hk, c.Hv, torch.bfloat16, torch.bfloat16)
    w = gdn.make_weights(c.conv_w, c.dt_bias, c.ssm_a, c.norm_w, device=dev)
    i = {k: getattr(c, k).to(dev) for k in ("x", "z")}
    hid, Wa, Wb = pc.hidden.to(dev), pc.W_a.to(dev), pc.W_b.to(dev)
    conv, S = c.conv0.to(dev), c.S0.to(dev)
    o = torch.empty(c.N, c.Hv * 128, device=dev, dtype=torch.bfloat16)
    am = timed_graph(lambda: gdn.gdn_decode_step_ab(d, w, i["x"], i["z"], hid, Wa, Wb, conv, S, o))
    ab = decode_bytes(c.N, c.Hk, c.Hv) + 2 * (c.N * 2048 + 2 * c.Hv * 2048) - 2 * 2 * c.N * c.Hv
    out["decode_B64_fold_ab_H2048"] = {"tokens_per_s": c.N / (am / 1e3), "us": 1e3 * am,
                                       "roofline": {"bound": "hbm", "achieved": ab / (am / 1e3) / 1e9, "peak": hbm,
                                                    "unit": "GB/s", "frac": ab / (am / 1e3) / 1e9 / hbm,
                                                    "algorithmic_bytes": ab}}
    del S, conv

    # the projections either side of the mixer: 27B dims over the T=8192 prefill (tensor-bound,
    # cuBLASLt) and, bound by reading the weights, the library's weight-streaming kernel at the
    # B=64 decode batch (35B and 27B dims) and the B=64 K=3 verify batch (35B dims)
    for name, T, H, Hk, Hv in (("proj_in_out_T8192_H5120", 8192, 5120, 16, 48),
                               ("proj_in_out_B64_H2048", 64, 2048, 16, 32),
                               ("proj_in_out_B64_H5120", 64, 5120, 16, 48),
                               ("proj_in_out_T192_H2048", 192, 2048, 16, 32)):
        c = gdn_inputs.make_proj_case(T=T, H=H, Hk=Hk, Hv=Hv, seed=7)
        d = gdn.make_dims(Hk, Hv, torch.bfloat16, torch.bfloat16)
        C, HvD = 128 * (2 * Hk + Hv), 128 * Hv
        ws = torch.empty(32 << 20, device=dev, dtype=torch.uint8)   # cuBLASLt's scratch (T > 256)
        t = {k: getattr(c, k).to(dev) for k in ("hidden", "W_qkv", "W_z", "W_a", "W_b", "y", "W_out")}
        bf = dict(device=dev, dtype=torch.bfloat16)
        x, z = torch.empty(T, C, **bf), torch.empty(T, HvD, **bf)
        a, b, po = torch.empty(T, Hv, **bf), torch.empty(T, Hv, **bf), torch.empty(T, H, **bf)

        def proj_in():
            gdn.gdn_in_proj(d, t["hidden"], t["W_qkv"], t["W_z"], t["W_a"], t["W_b"], x, z, a, b, workspace=ws)

        def proj_out():
            gdn.gdn_out_proj(d, t["y"], t["W_out"], po, workspace=ws)

        def proj():
            proj_in()
            proj_out()

        pm, pin, pout = timed_graph(proj), timed_graph(proj_in), timed_graph(proj_out)

        def torch_linear():   # the same five GEMMs through torch (cuBLAS), for comparison only
            for W, o in ((t["W_qkv"], x), (t["W_z"], z), (t["W_a"], a), (t["W_b"], b)):
                torch.matmul(t["hidden"], W.t(), out=o)
            torch.matmul(t["y"], t["W_out"].t(), out=po)

        cm = timed_graph(torch_linear)
        flops = 2.0 * T * H * (C + HvD + 2 * Hv) + 2.0 * T * HvD * H
        wbytes = 2 * H * (C + HvD + 2 * Hv) + 2 * H * HvD
        abytes = 2 * T * (H + C + HvD + 2 * Hv) + 2 * T * (HvD + H)
        out[name] = {"ms": pm, "in_ms": pin, "out_ms": pout, "torch_cublas_ms": cm,
                     "kernel": "weight-streaming (TMA + tcgen05)" if T <= 256 else "cuBLASLt",
                     "tflops": flops / (pm / 1e3) / 1e12,
                     "frac_of_bf16_peak": flops / (pm / 1e3) / 1e12 / tf,
                     "GBps": (wbytes + abytes) / (pm / 1e3) / 1e9,
                     "frac_of_hbm_peak": (wbytes + abytes) / (pm / 1e3) / 1e9 / hbm,
                     "flops": flops, "bytes": wbytes + abytes}
        del t, x, z, a, b, po, ws

    # packed varlen prefill, 8 sequences, T=65536
    c = gdn_inputs.varlen_t65536()
    d = gdn.make_dims(c.Hk, c.Hv, torch.bfloat16, torch.bfloat16)
    w = gdn.make_weights(c.conv_w, c.dt_bias, c.ssm_a, c.norm_w, device=dev)
    i = {k: getattr(c, k).to(dev) for k in ("x", "z", "a_raw", "b_raw")}
    cu_h = c.cu_seqlens.to(torch.int32)
    cu_d = cu_h.to(dev)
    conv0, S0 = c.conv0.to(dev), c.S0.to(dev)
    conv, S = conv0.clone(), S0.clone()
    po = torch.empty(c.T, c.Hv * 128, device=dev, dtype=torch.bfloat16)
    nws = gdn.gdn_prefill_workspace_bytes(d, c.N, c.T)
    ws = torch.empty(max(nws, 16), device=dev, dtype=torch.uint8)

    def call():
        conv.copy_(conv0)
        S.copy_(S0)
        e0.record(stream)
        gdn.gdn_prefill_chunked(d, w, cu_h, cu_d, i["x"], i["z"], i["a_raw"], i["b_raw"], conv, S, po,
                                zero_init=False, workspace=ws)
        e1.record(stream)

    ms = []
    for it in range(warmup + reps):
        flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        call()
        torch.cuda.synchronize()
        if it >= warmup:
            ms.append(e0.elapsed_time(e1))
    vm = statistics.mean(ms)
    vb = prefill_bytes(c.T, c.Hk, c.Hv, init_state=True, n_seq=c.N)
    out["prefill_varlen_N8_T65536"] = {"tokens_per_s": c.T / (vm / 1e3), "ms": vm,
                                       "lengths": [int(v) for v in (cu_h[1:] - cu_h[:-1])],
                                       "roofline": {"bound": "hbm", "achieved": vb / (vm / 1e3) / 1e9,
                                                    "peak": hbm, "unit": "GB/s",
                                                    "frac": vb / (vm / 1e3) / 1e9 / hbm,
                                                    "algorithmic_bytes": vb}}
    return out


def proj_part(dev):
    """The input and output projections at the B=64 decode batch, 35B dims (hidden 2048,
    16/32 heads), through the weight-streaming kernel (profiling aid)."""
    import gated_deltanet_linear_decode_gb300 as gdn
    T, H, Hk, Hv = 64, 2048, 16, 32
    c = gdn_inputs.make_proj_case(T=T, H=H, Hk=Hk, Hv=Hv, seed=7)
    d = gdn.make_dims(Hk, Hv, torch.bfloat16, torch.bfloat16)
    t = {k: getattr(c, k).to(dev) for k in ("hidden", "W_qkv", "W_z", "W_a", "W_b", "y", "W_out")}
    bf = dict(device=dev, dtype=torch.bfloat16)
    x, z = torch.empty(T, 128 * (2 * Hk + Hv), **bf), torch.empty(T, 128 * Hv, **bf)
    a, b, po = torch.empty(T, Hv, **bf), torch.empty(T, Hv, **bf), torch.empty(T, H, **bf)
    def run():
        gdn.gdn_in_proj(d, t["hidden"], t["W_qkv"], t["W_z"], t["W_a"], t["W_b"], x, z, a, b)
        gdn.gdn_out_proj(d, t["y"], t["W_out"], po)
    return run


def decode_bf16_part(dev):
    """The B=64 decode step (16/32 heads) with the state stored as bf16, as timed in `extras`."""
    import gated_deltanet_linear_decode_gb300 as gdn
    c = gdn_inputs.decode_b64()
    d = gdn.make_dims(c.Hk, c.Hv, torch.bfloat16, torch.bfloat16, state_dtype=torch.bfloat16)
    w = gdn.make_weights(c.conv_w, c.dt_bias, c.ssm_a, c.norm_w, device=dev)
    i = {k: getattr(c, k).to(dev) for k in ("x", "z", "a_raw", "b_raw")}
    conv, S = c.conv0.to(dev), c.S0.to(dev).to(torch.bfloat16)
    o = torch.empty(c.N, c.Hv * 128, device=dev, dtype=torch.bfloat16)
    return lambda: gdn.gdn_decode_step(d, w, i["x"], i["z"], i["a_raw"], i["b_raw"], conv, S, o)


def varlen_part(dev):
    """The packed varlen prefill (8 sequences, T=65536, nonzero initial state), as timed in `extras`."""
    import gated_deltanet_linear_decode_gb300 as gdn
    c = gdn_inputs.varlen_t65536()
    d = gdn.make_dims(c.Hk, c.Hv, torch.bfloat16, torch.bfloat16)
    w = gdn.make_weights(c.conv_w, c.dt_bias, c.ssm_a, c.norm_w, device=dev)
    i = {k: getattr(c, k).to(dev) for k in ("x", "z", "a_raw", "b_raw")}
    cu_h = c.cu_seqlens.to(torch.int32)
    cu_d = cu_h.to(dev)
    conv, S = c.conv0.to(dev), c.S0.to(dev)
    po = torch.empty(c.T, c.Hv * 128, device=dev, dtype=torch.bfloat16)
    ws = torch.empty(max(gdn.gdn_prefill_workspace_bytes(d, c.N, c.T), 16), device=dev, dtype=torch.uint8)
    return lambda: gdn.gdn_prefill_chunked(d, w, cu_h, cu_d, i["x"], i["z"], i["a_raw"], i["b_raw"], conv, S, po,
                                           zero_init=False, workspace=ws)


def run_part(args):
    """Warm-up then timed launches of one part only (profiling aid)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = Workload(dev, args.prefill_tokens)
    fn = {"prefill": wl.prefill, "decode": wl.decode, "verify": wl.verify}.get(args.only)
    if args.only == "proj":
        fn = proj_part(dev)
    elif args.only == "decode-bf16":
        fn = decode_bf16_part(dev)
    elif args.only == "varlen":
        fn = varlen_part(dev)
    for _ in range(args.warmup + args.steps):
        wl.flush_l2()
        fn()
    torch.cuda.synchronize()
    print(f"ran {args.only}: {args.warmup} warm-up + {args.steps} launches", flush=True)


def _barrier(world):
    if world > 1:
        torch.distributed.barrier()


def _max_over_ranks(v, world):
    if world <= 1:
        return v
    # NCCL reduces device tensors; the CPU (gloo) process group used by the tests reduces host ones
    on_gpu = torch.distributed.get_backend() == "nccl"
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if on_gpu else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ the oracle (CPU)
def oracle_step(cases, prefill_tokens=None, n_threads=0):
    """One step of the workload through the CPU oracle (fp64, OpenMP): the
    prefill (all 48 heads; only its first `prefill_tokens` tokens when given),
    the B=64 decode step and the B=64 K=3 verify walk with checkpoints.
    Returns the seconds of (prefill, decode, verify)."""
    import oracle
    pc, dc, vc = cases
    n = pc.T if prefill_tokens is None else prefill_tokens
    t0 = time.perf_counter()
    oracle.forward(pc.Hk, pc.Hv, pc.x[:n], pc.z[:n], pc.a_raw[:n], pc.b_raw[:n], pc.conv_w, pc.dt_bias, pc.ssm_a,
                   pc.norm_w, pc.conv0, pc.S0, cu_seqlens=[0, n], n_threads=n_threads)
    t1 = time.perf_counter()
    oracle.forward(dc.Hk, dc.Hv, dc.x, dc.z, dc.a_raw, dc.b_raw, dc.conv_w, dc.dt_bias, dc.ssm_a, dc.norm_w,
                   dc.conv0, dc.S0, cu_seqlens=np.arange(dc.N + 1), n_threads=n_threads)
    t2 = time.perf_counter()
    oracle.verify_checkpoints(vc.Hk, vc.Hv, vc.x, vc.z, vc.a_raw, vc.b_raw, vc.conv_w, vc.dt_bias, vc.ssm_a,
                              vc.norm_w, vc.conv0, vc.S0, vc.K, n_threads=n_threads)
    t3 = time.perf_counter()
    return t1 - t0, t2 - t1, t3 - t2


def host_cores():
    """CPU cores this process may run on, and the oracle's OpenMP thread count."""
    import oracle
    return len(os.sched_getaffinity(0)), oracle.max_threads()


def single_thread_rates(cases, prefill_tokens=256):
    """The oracle on one thread, per part of the step: the B=64 decode and the
    B=64 K=3 verify whole, the prefill on its first `prefill_tokens` tokens."""
    pc, dc, vc = cases
    tp, td, tv = oracle_step(cases, prefill_tokens, n_threads=1)
    return {"prefill_tokens_per_s": prefill_tokens / tp, "decode_tokens_per_s": dc.N / td,
            "verify_tokens_per_s": vc.N * vc.K / tv,
            "sample": f"one thread: prefill tokens 0..{prefill_tokens - 1} of T=8192 (48 heads), the whole B=64 "
                      f"decode, the whole B=64 K=3 verify"}


def cpu_baseline(min_seconds=10.0):
    """The oracle, as it stands, on the host cores: whole steps of the workload,
    repeated until at least `min_seconds` of CPU work; and its single-thread
    rates on a bounded sample."""
    import oracle
    oracle.build()
    cases = (gdn_inputs.prefill_t8192(), gdn_inputs.decode_b64(), gdn_inputs.verify_b64_k3())
    tok = cases[0].T + cases[1].N + cases[2].N * cases[2].K
    reps, used = 0, 0.0
    while used < min_seconds or reps == 0:
        used += sum(oracle_step(cases))
        reps += 1
    cores, omp = host_cores()
    return {"value": tok * reps / used, "unit": "tokens/s", "cores": omp, "cores_available": cores,
            "kind": "oracle",
            "sample": f"fp64 C oracle, whole steps of the workload (prefill T=8192 all 48 heads + B=64 decode + "
                      f"B=64 K=3 verify) x{reps}, {used:.1f} s of CPU work, {omp} OpenMP threads on {cores} cores",
            "seconds": used, "single_thread": single_thread_rates(cases)}


def step_config(world):
    """The workload description both arms print."""
    return {"workload": WORKLOAD, "tokens_per_step": TOKENS_PER_STEP,
            "l2": "flushed (256 MiB write) before each timed step; inputs also exceed L2",
            "parallelism": f"replicas x{world}"}


def run_reference(args, rank, world):
    """The reference arm: the fp64 oracle as it stands on the host cores, timing
    whole steps of the workload (no extrapolation)."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    cases = (gdn_inputs.prefill_t8192(), gdn_inputs.decode_b64(), gdn_inputs.verify_b64_k3())
    tok = cases[0].T + cases[1].N + cases[2].N * cases[2].K
    for _ in range(args.warmup):
        oracle_step(cases)
    times = [sum(oracle_step(cases)) for _ in range(args.steps)]
    tot = sum(times)
    value = tok * len(times) / tot
    cores, omp = host_cores()
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; no weights or dataset)", "config": step_config(world),
        "cpu_baseline": {"kind": "oracle", "cores": omp, "cores_available": cores, "value": value,
                         "unit": "tokens/s",
                         "sample": f"whole steps of the workload (prefill T=8192 all 48 heads + B=64 decode + B=64 K=3 "
                                   f"verify), {args.steps} timed after {args.warmup} untimed, {omp} OpenMP threads on "
                                   f"{cores} cores"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gdn", choices=["gdn", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the batch-1 graph decode and the varlen T=65536 prefill (timed outside the step)")
    ap.add_argument("--prefill-tokens", type=int, default=8192,
                    help="with --only prefill: the sequence length (a smaller case for profiling)")
    ap.add_argument("--only", choices=["prefill", "decode", "verify", "proj", "decode-bf16", "varlen"], default=None,
                    help="run only one part of the step (for profiling); no JSON line")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if args.only:
        run_part(args)
        return
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group("nccl")
    line = run_gpu(args, rank, world)
    if rank == 0 and not args.no_extras:
        line["extras"] = run_extras(torch.device("cuda", torch.cuda.current_device()), max(args.warmup, 1),
                                    max(1, min(args.steps, 5)))
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline()
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
