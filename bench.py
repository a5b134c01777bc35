#!/usr/bin/env python
"""Benchmark of the fused per-token decoder path on GB300.

One step = one pass of the whole hot path at its configured shapes:
  * rmsnorm       x [512, D], D in {128, 512, 1024, 1536, 2048, 2176, 4096, 8192},
                  in fp32, fp16 and bf16 (24 launches)
  * add_rmsnorm   x, res [T, 1536] bf16, T in {1, 16, 256, 4096} (4 launches)
  * rope_kv_store Qwen2.5-1.5B GQA, T in {1, 64, 2048}, cache [2, 4096, 16, 2, 128] (3 launches)
  * swiglu/reglu  gate_up [T, 2 x 14336] bf16, T in {1, 64, 512, 4096} (8 launches)
  * decode chain  28 layers x (add_rmsnorm, rope_kv_store, add_rmsnorm, swiglu) at
                  batch 1 and 64 (Qwen2.5-1.5B shapes), each replayed from a CUDA graph
                  (2 x 112 launches)
Every input is synthetic and seeded, resident in HBM before timing. L2 is
flushed before every step (a 256 MiB write, then a read, so no dirty lines are
left to write back inside the step). Each step is queued behind a short
device-side delay so the host has enqueued the whole step before the GPU starts
it; the timed region is the step alone (CUDA events on the launching stream),
with one more event pair around the dominant kernel (the largest stream).
Kernels are launched with programmatic dependent launch (--no-pdl turns it
off). `value` = algorithmic bytes of the step / device time of the step, summed
over ranks (each rank runs its own replica: weak scaling).

Also measured, per kernel: the time of one launch alone (clean L2, one event
pair: includes the event overhead) and the streaming rate (back-to-back
launches over rotating copies of its buffers that exceed 4x L2, so every launch
reads cold data, replayed from a CUDA graph so the host's enqueue rate cannot pace
them) with its GB/s and fraction of the measured HBM peak, and the fraction of
the launch's floor in a dependent chain (its bytes at that peak plus the measured
per-launch latency) that it reaches; rows/s
at decode batch; the launch latency of the smallest launches; row-scaled companion shapes (>= 256 MB of traffic), an
end-to-end number through the same C ABI from pinned host buffers, and the CPU
oracle on a bounded sample of the same step (rank 0, one GPU only).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
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

METRIC = "achieved HBM GB/s and % of GB300 peak per kernel; rows/s at decode batch"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
STREAM_BYTES = 512 << 20   # per-kernel streaming measurement: total bytes over the rotating copies
NVTX_STEP = "sra_timed_step"
WORKLOAD = ("decoder per-token hot path at the configured shapes: rmsnorm 512xD sweep (8 widths x fp32/fp16/bf16), "
            "add_rmsnorm bf16 Tx1536 T={1,16,256,4096}, rope_kv_store Qwen2.5-1.5B GQA T={1,64,2048}, "
            "swiglu+reglu Llama-3-8B gate_up T={1,64,512,4096}, 28-layer decode chain B={1,64}")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["sra", "reference"], default="sra")
    p.add_argument("--only", default="", help="comma list of entry-name prefixes to run (profiling)")
    p.add_argument("--no-chain", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-companions", action="store_true")
    p.add_argument("--no-pdl", action="store_true", help="launch without programmatic dependent launch")
    p.add_argument("--sweep-variants", action="store_true",
                   help="A/B: time every RMSNorm / GLU variant on every norm / GLU shape (prints its own JSON)")
    p.add_argument("--force", default="",
                   help="comma list op=variant applied with sra_force_variant before anything runs (profiling A/B)")
    p.add_argument("--sweep-cps", action="store_true",
                   help="with --sweep-variants: also cap the register RMSNorm variants at 1-6 CTAs per SM")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU-baseline duration")
    return p.parse_args()


# --------------------------------------------------------------------------- workload
class Entry:
    """One launch of the step: a raw C-ABI call with fixed arguments."""

    def __init__(self, name, op, bytes_, rows, fn, args, inputs=(), outputs=(), dtype="bf16", keep=()):
        self.name, self.op, self.bytes, self.rows = name, op, bytes_, rows
        self.keep = keep   # every tensor whose raw pointer is in `args` stays alive with the entry
        self.fn, self.args = fn, args
        self.inputs, self.outputs = list(inputs), list(outputs)   # device tensors fed / produced per step
        self.dtype = dtype
        self.times = []

    def launch(self):
        st = self.fn(*self.args)
        if st != 0:
            raise RuntimeError(f"{self.name}: status {st}")

    def tensors(self):
        k = self.keep
        if isinstance(k, dict):
            return list(k.values())
        if isinstance(k, (list, tuple)):
            return list(k)
        return [k]

    def replicas(self, n, stream_handle=None):
        """n launch closures, each on its own device copy of every buffer the launch touches
        (and, if given, on another stream: the stream is every call's last argument)."""
        import torch

        out = []
        for _ in range(n):
            remap, hold = {}, []
            for t in self.tensors():
                c = torch.empty_like(t)
                c.copy_(t)
                remap[t.data_ptr()] = c.data_ptr()
                hold.append(c)
            args = tuple(remap.get(a, a) if isinstance(a, int) and not isinstance(a, bool) else a
                         for a in self.args)
            if stream_handle is not None:
                args = args[:-1] + (stream_handle,)
            fn = self.fn

            def call(args=args, hold=hold):
                st = fn(*args)
                if st != 0:
                    raise RuntimeError(f"{self.name}: status {st}")

            out.append(call)
        return out


def build_entries(dev, stream_handle, only=(), companions=False):
    import torch

    import swiglu_rmsnorm_add_gb300 as sra
    from swiglu_rmsnorm_add_gb300 import synthetic as syn

    L = sra.lib()
    code = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
    short = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}
    entries = []

    def want(name):
        return not only or any(name.startswith(o) for o in only)

    if not companions:
        for dt in (torch.float32, torch.float16, torch.bfloat16):
            for D in syn.RMS_SWEEP_D:
                name = f"rmsnorm:{short[dt]}:512x{D}"
                if not want(name):
                    continue
                x, w = syn.rms_inputs(512, D, dt, 1001)
                x, w = x.to(dev), w.to(dev)
                out = torch.empty_like(x)
                s = x.element_size()
                entries.append(Entry(name, "rmsnorm", 2 * 512 * D * s + D * s, 512, L.sra_rmsnorm,
                                     (x.data_ptr(), w.data_ptr(), out.data_ptr(), 512, D, D, D, syn.EPS, code[dt],
                                      stream_handle), [x], [out], short[dt], keep=(x, w, out)))
        Ts_add, Ts_rope, Ts_glu = syn.ADD_RMS_T, syn.ROPE_T, syn.GLU_T
    else:
        Ts_add, Ts_rope, Ts_glu = (32768,), (32768,), ()
        # row-scaled companions of the RMSNorm widths: the Qwen2.5-1.5B hidden row in bf16, and
        # the fp32 rows of 8192 and 4096 whose 512-row configured shapes are dominated by the
        # fixed cost of a launch (>= 256 MB each, so they show the streaming rate)
        for dt, R, D in ((torch.bfloat16, 65536, 1536), (torch.float32, 4096, 8192), (torch.float32, 8192, 4096)):
            name = f"rmsnorm:{short[dt]}:{R}x{D}"
            if want(name):
                x, w = syn.rms_inputs(R, D, dt, 1001)
                x, w = x.to(dev), w.to(dev)
                out = torch.empty_like(x)
                s = x.element_size()
                entries.append(Entry(name, "rmsnorm", 2 * R * D * s + D * s, R, L.sra_rmsnorm,
                                     (x.data_ptr(), w.data_ptr(), out.data_ptr(), R, D, D, D, syn.EPS, code[dt],
                                      stream_handle), [x], [out], short[dt], keep=(x, w, out)))
    for T in Ts_add:
        name = f"add_rmsnorm:bf16:{T}x1536"
        if not want(name):
            continue
        x, r, w = syn.add_rms_inputs(T, 1536, torch.bfloat16, 1001)
        x, r, w = x.to(dev), r.to(dev), w.to(dev)
        out = torch.empty_like(x)
        entries.append(Entry(name, "add_rmsnorm", 4 * T * 1536 * 2 + 1536 * 2, T, L.sra_add_rmsnorm,
                             (x.data_ptr(), r.data_ptr(), w.data_ptr(), out.data_ptr(), T, 1536, 1536, 1536, 1536,
                              syn.EPS, 2, stream_handle), [x, r], [x, out], keep=(x, r, w, out)))
    tables = None
    # (style, Q/K UClip fused, T): the neox shapes of the step; the interleaved (GPT-J) pairing
    # and the fused Q/K norm as companions
    ropes = [(0, False, T) for T in Ts_rope]
    if companions:
        ropes += [(1, False, 2048), (1, False, 32768), (0, True, 2048), (0, True, 32768)]
    for style, qk, T in ropes:
        kind = ("rope_kv_store" if style == 0 else "rope_kv_store_interleaved") + ("_qk_uclip" if qk else "")
        name = f"{kind}:bf16:T{T}"
        if not want(name):
            continue
        if tables is None:
            tables = syn.rope_tables(32768, 128, 1e6)
        nb = max(4096, (T + 15) // 16)
        inp = {k: v.to(dev) for k, v in syn.rope_inputs(T, 1002, num_blocks=nb, tables=tables).items()}
        per_tok = 2 * 12 * 128 * 2 + 2 * 128 * 2 * 2 + 2 * 64 * 4 + 16 + 2 * 2 * 128 * 2
        common = (inp["q"].data_ptr(), inp["k"].data_ptr(), inp["v"].data_ptr(), inp["cos"].data_ptr(),
                  inp["sin"].data_ptr(), inp["pos"].data_ptr(), inp["slot_mapping"].data_ptr(),
                  inp["kv_cache"].data_ptr(), T, 12, 2, 128, 12 * 128, 2 * 128, 2 * 128, 32768, nb, 16, None, style)
        if qk:
            params = [p.to(dev) for i in range(4) for p in (syn.uclip_params(128, True, True, 1002 + i)[i % 2],)]
            inp = dict(inp, **{f"p{i}": p for i, p in enumerate(params)})
            fn, args = L.sra_rope_kv_store_qk_uclip, common + tuple(p.data_ptr() for p in params) + (-1.0, 1.0)
            nbytes = per_tok * T + 4 * 128 * 4
        else:
            fn, args, nbytes = L.sra_rope_kv_store_ex, common, per_tok * T
        entries.append(Entry(name, "rope_kv_store", nbytes, T, fn, args + (2, stream_handle),
                             [inp["q"], inp["k"], inp["v"], inp["pos"], inp["slot_mapping"]], [inp["q"]],
                             keep=inp))
    if companions:
        # UClip / DyHT: in place of the hidden-row RMSNorm (scalar alpha, per-channel gamma),
        # and the Q-head norm in place on a fused QKV buffer (per-channel alpha and gamma)
        for T in (4096, 65536):
            name = f"dyht:bf16:{T}x1536"
            if not want(name):
                continue
            x = syn.normal((T, 1536), 0.0, 1.0, torch.bfloat16, 1005, 1).to(dev)
            a, g = (p.to(dev) for p in syn.uclip_params(1536, False, True, 1005))
            out = torch.empty_like(x)
            entries.append(Entry(name, "uclip", 2 * T * 1536 * 2 + 1536 * 4 + 4, T, L.sra_uclip,
                                 (x.data_ptr(), a.data_ptr(), g.data_ptr(), out.data_ptr(), T, 1, 1536, 1536, 1536,
                                  1536, 1536, 0, 1, -1.0, 1.0, 2, stream_handle), [x], [out], keep=(x, a, g, out)))
        T = 32768
        name = f"uclip_q:bf16:T{T}"
        if want(name):
            qkv = syn.qkv_inputs(T, 12, 2, 128, torch.bfloat16, 1006).to(dev)
            a, g = (p.to(dev) for p in syn.uclip_params(128, True, True, 1006))
            W = 16 * 128
            entries.append(Entry(name, "uclip", 2 * T * 12 * 128 * 2 + 2 * 128 * 4, T * 12, L.sra_uclip,
                                 (qkv.data_ptr(), a.data_ptr(), g.data_ptr(), qkv.data_ptr(), T, 12, 128, W, 128, W,
                                  128, 1, 1, -1.0, 1.0, 2, stream_handle), [qkv], [qkv], keep=(qkv, a, g)))
    if companions:
        # decode attention over the paged cache (Qwen2.5-1.5B heads): the read side of rope_kv_store
        for B, ctx in ((1, 32768), (32, syn.ATTN_CTX), (64, syn.ATTN_CTX)):
            name = f"decode_attention:bf16:B{B}xctx{ctx}"
            if not want(name):
                continue
            nb = max(4096, B * ((ctx + 15) // 16))
            q, cache, table, seq = (t.to(dev) for t in syn.attention_inputs(B, ctx, 12, 2, 128, 16, nb,
                                                                             torch.bfloat16, 1012))
            out = torch.empty_like(q)
            nblk = (ctx + 15) // 16
            nbytes = 2 * B * ctx * 2 * 128 * 2 + 2 * B * 12 * 128 * 2 + 4 * (B * nblk + B)
            entries.append(Entry(name, "decode_attention", nbytes, B, L.sra_paged_decode_attention,
                                 (q.data_ptr(), cache.data_ptr(), table.data_ptr(), seq.data_ptr(), out.data_ptr(),
                                  B, 12, 2, 128, 12 * 128, 12 * 128, nb, 16, table.shape[1], 128 ** -0.5, None, 2,
                                  stream_handle), [q, table, seq], [out], keep=(q, cache, table, seq, out)))
        # few (request, kv head) pairs over a long context: split over up to one CTA per SM, the
        # partials merged through a caller workspace
        for B, ctx in ((1, 32768), (2, 16384)):
            name = f"decode_attention_ws:bf16:B{B}xctx{ctx}"
            if not want(name):
                continue
            nb = max(4096, B * ((ctx + 15) // 16))
            q, cache, table, seq = (t.to(dev) for t in syn.attention_inputs(B, ctx, 12, 2, 128, 16, nb,
                                                                             torch.bfloat16, 1013))
            out = torch.empty_like(q)
            ws = sra.decode_attention_workspace(B, 12, 2, 128, table.shape[1], 16, torch.bfloat16, dev)
            if ws is None:
                raise RuntimeError(f"{name}: the shape takes no workspace split")
            nblk = (ctx + 15) // 16
            nbytes = 2 * B * ctx * 2 * 128 * 2 + 2 * B * 12 * 128 * 2 + 4 * (B * nblk + B)
            entries.append(Entry(name, "decode_attention", nbytes, B, L.sra_paged_decode_attention_ws,
                                 (q.data_ptr(), cache.data_ptr(), table.data_ptr(), seq.data_ptr(), out.data_ptr(),
                                  B, 12, 2, 128, 12 * 128, 12 * 128, nb, 16, table.shape[1], 128 ** -0.5,
                                  ws.data_ptr(), ws.numel(), None, 2, stream_handle), [q, table, seq], [out],
                                 keep=(q, cache, table, seq, out, ws)))
    if companions:
        # RMSNorm / SwiGLU fused into the projection they feed (Qwen2.5-1.5B: ln1 + qkv_proj,
        # silu(gate) * up + down_proj), decode batch 1 and 64
        for B in (1, 64):
            K, N = syn.QWEN25_QKV["K"], syn.QWEN25_QKV["N"]
            name = f"rmsnorm_linear:bf16:B{B}x{K}x{N}"
            if want(name):
                x = syn.normal((B, K), 0.0, 1.0, torch.bfloat16, 1030, 1).to(dev)
                w = syn.normal((K,), 1.0, 0.1, torch.bfloat16, 1030, 2).to(dev)
                W = syn.linear_weight(N, K, torch.bfloat16, 1030).to(dev)
                y = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
                nbytes = (N * K + B * K + K + B * N) * 2
                entries.append(Entry(name, "linear", nbytes, B, L.sra_rmsnorm_linear,
                                     (x.data_ptr(), w.data_ptr(), W.data_ptr(), y.data_ptr(), B, K, N, K, N, syn.EPS,
                                      2, stream_handle), [x], [y], keep=(x, w, W, y)))
            name = f"rmsnorm_linear_ws:bf16:B{B}x{K}x{N}"
            if B >= 32 and want(name):
                x = syn.normal((B, K), 0.0, 1.0, torch.bfloat16, 1030, 1).to(dev)
                w = syn.normal((K,), 1.0, 0.1, torch.bfloat16, 1030, 2).to(dev)
                W = syn.linear_weight(N, K, torch.bfloat16, 1030).to(dev)
                y = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
                ws = sra.linear_workspace(B, K, torch.bfloat16, dev, N)
                nbytes = (N * K + B * K + K + B * N) * 2
                entries.append(Entry(name, "linear", nbytes, B, L.sra_rmsnorm_linear_ws,
                                     (x.data_ptr(), w.data_ptr(), W.data_ptr(), y.data_ptr(), B, K, N, K, N, syn.EPS,
                                      ws.data_ptr(), ws.numel() * 2, 2, stream_handle), [x], [y],
                                     keep=(x, w, W, y, ws)))
            I, N = syn.QWEN25_DOWN["I"], syn.QWEN25_DOWN["N"]
            name = f"swiglu_linear_ws:bf16:B{B}x{I}x{N}"
            if B >= 32 and want(name):
                gu = syn.normal((B, 2 * I), 0.0, 1.0, torch.bfloat16, 1031, 3).to(dev)
                W = syn.linear_weight(N, I, torch.bfloat16, 1031).to(dev)
                y = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
                ws = sra.linear_workspace(B, I, torch.bfloat16, dev, N)
                nbytes = (N * I + B * 2 * I + B * N) * 2
                entries.append(Entry(name, "linear", nbytes, B, L.sra_glu_linear_ws,
                                     (gu.data_ptr(), W.data_ptr(), y.data_ptr(), B, I, N, 2 * I, N, 0, ws.data_ptr(),
                                      ws.numel() * 2, 2, stream_handle), [gu], [y], keep=(gu, W, y, ws)))
            name = f"swiglu_linear:bf16:B{B}x{I}x{N}"
            if want(name):
                gu = syn.normal((B, 2 * I), 0.0, 1.0, torch.bfloat16, 1031, 3).to(dev)
                W = syn.linear_weight(N, I, torch.bfloat16, 1031).to(dev)
                y = torch.empty(B, N, dtype=torch.bfloat16, device=dev)
                nbytes = (N * I + B * 2 * I + B * N) * 2
                entries.append(Entry(name, "linear", nbytes, B, L.sra_glu_linear,
                                     (gu.data_ptr(), W.data_ptr(), y.data_ptr(), B, I, N, 2 * I, N, 0, 2,
                                      stream_handle), [gu], [y], keep=(gu, W, y)))
    if companions:
        # the decode chain's own batch-64 shapes, standalone (Qwen2.5-1.5B: hidden 1536, intermediate 8960)
        name = "add_rmsnorm:bf16:64x1536"
        if want(name):
            x, r, w = syn.add_rms_inputs(64, 1536, torch.bfloat16, 1004)
            x, r, w = x.to(dev), r.to(dev), w.to(dev)
            out = torch.empty_like(x)
            entries.append(Entry(name, "add_rmsnorm", 4 * 64 * 1536 * 2 + 1536 * 2, 64, L.sra_add_rmsnorm,
                                 (x.data_ptr(), r.data_ptr(), w.data_ptr(), out.data_ptr(), 64, 1536, 1536, 1536,
                                  1536, syn.EPS, 2, stream_handle), [x, r], [x, out], keep=(x, r, w, out)))
        I5 = syn.QWEN25_DOWN["I"]
        name = f"swiglu:bf16:64x{I5}"
        if want(name):
            gu = syn.glu_inputs(64, I5, torch.bfloat16, 1004).to(dev)
            out = torch.empty(64, I5, dtype=torch.bfloat16, device=dev)
            entries.append(Entry(name, "swiglu", 64 * (2 * I5 * 2 + I5 * 2), 64, L.sra_glu,
                                 (gu.data_ptr(), out.data_ptr(), 64, I5, 2 * I5, I5, 0, 2, stream_handle), [gu],
                                 [out], keep=(gu, out)))
    I = syn.LLAMA3_8B_MLP["intermediate"]
    for T in Ts_glu:
        gu = None
        for act, an in ((0, "swiglu"), (1, "reglu")):
            name = f"{an}:bf16:{T}x{I}"
            if not want(name):
                continue
            if gu is None:
                gu = syn.glu_inputs(T, I, torch.bfloat16, 1003).to(dev)
            out = torch.empty(T, I, dtype=torch.bfloat16, device=dev)
            entries.append(Entry(name, an, T * (2 * I * 2 + I * 2), T, L.sra_glu,
                                 (gu.data_ptr(), out.data_ptr(), T, I, 2 * I, I, act, 2, stream_handle),
                                 [gu] if act == 0 else [], [out], keep=(gu, out)))
    return entries


class ChainEntry:
    def __init__(self, B, dev, pdl=True):
        from swiglu_rmsnorm_add_gb300.chain import DecodeChain

        self.name = f"chain:bf16:B{B}x28"
        self.op = "chain"
        self.B = B
        self.rows = B
        self.chain = DecodeChain(B, device=dev)
        self.chain.capture(pdl=pdl)
        self.bytes_by_kind = self.chain.bytes_per_step()
        self.bytes = sum(self.bytes_by_kind.values())
        self.times = []
        self.dtype = "bf16"
        c = self.chain
        self.inputs = [c.pos] + [lay["slots"] for lay in c.layers]
        self.outputs = [c.x]

    def launch(self):
        self.chain.replay()


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- helpers
def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 copy measurement)"


def kernel_traffic(entry_name):
    """dram read+write bytes per launch from the committed ncu summary, if the kernel is unchanged."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    rec = table.get(entry_name)
    if not rec:
        return None
    h = hashlib.sha256()
    for src in rec.get("sources", []):
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != rec.get("sources_sha256"):
        return None
    return rec.get("dram_bytes_per_launch")


def reduce_max(x: float, device) -> float:
    """The maximum of x over all ranks (x itself when not distributed)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_value(bytes_per_rank_step: int, ms_max: float, world: int) -> float:
    """Whole-job GB/s of a weak-scaling step: every rank moves the same bytes; the
    slowest rank's step time sets the pace."""
    return world * bytes_per_rank_step / (ms_max / 1e3) / 1e9


def dist_setup(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# --------------------------------------------------------------------------- CPU oracle
_PLAN_CACHE: dict = {}


def cpu_sample_run(target_seconds, threads=None, fraction=None):
    """Run the CPU oracle over a row-subsampled copy of one step; returns a cpu_baseline dict.

    Rows (tokens) of every launch of the step are subsampled by the same
    fraction; the chain contributes its per-layer kernels on subsampled batch
    rows. Work is split over `threads` Python threads (each ctypes call releases
    the GIL), so the oracle itself stays single-threaded plain C++.
    """
    import concurrent.futures as cf

    import torch

    import oracle
    from swiglu_rmsnorm_add_gb300 import synthetic as syn

    threads = threads or os.cpu_count() or 1
    I = syn.LLAMA3_8B_MLP["intermediate"]
    jobs = _PLAN_CACHE.setdefault("jobs", [])   # (bytes, thunk)

    def rows_of(n, frac):
        return max(1, int(round(n * frac)))

    def plan(frac):
        if _PLAN_CACHE.get("frac") == frac and jobs:
            return
        _PLAN_CACHE["frac"] = frac
        jobs.clear()
        for dt in (torch.float32, torch.float16, torch.bfloat16):
            for D in syn.RMS_SWEEP_D:
                r = rows_of(512, frac)
                x, w = syn.rms_inputs(r, D, dt, 1001)
                out = torch.empty_like(x)
                jobs.append((2 * r * D * x.element_size() + D * x.element_size(),
                             lambda x=x, w=w, out=out: oracle.rmsnorm(x, w, out, syn.EPS)))
        for T in syn.ADD_RMS_T:
            r = rows_of(T, frac)
            x, res, w = syn.add_rms_inputs(r, 1536, torch.bfloat16, 1001)
            out = torch.empty_like(x)
            jobs.append((4 * r * 1536 * 2 + 3072, lambda x=x, res=res, w=w, out=out:
                         oracle.add_rmsnorm(x, res, w, out, syn.EPS)))
        tables = syn.rope_tables(32768, 128, 1e6)
        for T in syn.ROPE_T:
            r = rows_of(T, frac)
            inp = syn.rope_inputs(r, 1002, tables=tables, num_blocks=max(1, (r + 15) // 16))
            jobs.append((8720 * r, lambda inp=inp: oracle.rope_kv_store(**inp)))
        for T in syn.GLU_T:
            r = rows_of(T, frac)
            gu = syn.glu_inputs(r, I, torch.bfloat16, 1003)
            for act in ("silu", "relu"):
                out = torch.empty(r, I, dtype=torch.bfloat16)
                jobs.append((86016 * r, lambda gu=gu, out=out, act=act: oracle.glu(gu, out, act)))
        for B in (1, 64):
            r = rows_of(B, frac)
            x, res, w = syn.add_rms_inputs(r, 1536, torch.bfloat16, 1004)
            gu = syn.glu_inputs(r, 8960, torch.bfloat16, 1004)
            inp = syn.rope_inputs(r, 1004, tables=tables, num_blocks=max(1, (r + 15) // 16))
            for _ in range(28):
                out = torch.empty_like(x)
                jobs.append((4 * r * 1536 * 2 + 3072, lambda x=x, res=res, w=w, out=out:
                             oracle.add_rmsnorm(x, res, w, out, syn.EPS)))
                jobs.append((8720 * r, lambda inp=inp: oracle.rope_kv_store(**inp)))
                jobs.append((4 * r * 1536 * 2 + 3072, lambda x=x, res=res, w=w, out=out:
                             oracle.add_rmsnorm(x, res, w, out, syn.EPS)))
                o2 = torch.empty(r, 8960, dtype=torch.bfloat16)
                jobs.append((r * 8960 * 6, lambda gu=gu, o2=o2: oracle.swiglu(gu, o2)))

    def run():
        t0 = time.perf_counter()
        with cf.ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda j: j[1](), sorted(jobs, key=lambda j: -j[0])))
        return time.perf_counter() - t0

    if fraction is None:
        plan(1 / 64)          # calibrate on a small sample
        dt = run()
        b = sum(j[0] for j in jobs)
        rate = b / max(dt, 1e-6)
        full = 1.04e9 + 2.6e6 + 156e6      # approx algorithmic bytes of one full step
        fraction = min(1.0, max(1 / 512, target_seconds * rate / full))
    plan(fraction)
    dt = run()
    b = sum(j[0] for j in jobs)
    return {"value": b / dt / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"every launch of one step with rows/tokens subsampled to {fraction:.4f} of the step "
                      f"({b / 1e6:.1f} MB algorithmic, {dt:.1f} s wall, {threads} threads over row chunks)",
            "seconds": dt, "bytes": b, "fraction": fraction}


def cpu_rows_run():
    """The oracle timed beside each widened row (one thread, a small sample of the row's
    companion workload); returns {companion name prefix: {"gbs", "bytes", "seconds", "sample"}}."""
    import torch

    import oracle
    from swiglu_rmsnorm_add_gb300 import synthetic as syn

    tables = syn.rope_tables(32768, 128, 1e6)
    out = {}

    def timed(name, nbytes, sample, fn):
        n, t0 = 0, time.perf_counter()
        while True:  # repeat the sample for at least a quarter of a second
            fn()
            n += 1
            dt = time.perf_counter() - t0
            if dt >= 0.25:
                break
        out[name] = {"gbs": round(n * nbytes / dt / 1e9, 4), "bytes": n * nbytes, "seconds": round(dt, 3),
                     "sample": f"{sample}, {n} runs"}

    T = 256
    inp = syn.rope_inputs(T, 1002, tables=tables, num_blocks=64)
    timed("rope_kv_store_interleaved", 8720 * T, f"T={T}", lambda: oracle.rope_kv_store(**inp, style="interleaved"))
    inp = syn.rope_inputs(T, 1002, tables=tables, num_blocks=64)
    ps = tuple(syn.uclip_params(128, True, True, 1002 + i)[i % 2] for i in range(4))
    timed("rope_kv_store_qk_uclip", 8720 * T, f"T={T}",
          lambda: oracle.qk_uclip_rope_kv_store(inp["q"], inp["k"], inp["v"], inp["cos"], inp["sin"], inp["pos"],
                                                inp["slot_mapping"], inp["kv_cache"], *ps))
    x = syn.normal((512, 1536), 0.0, 1.0, torch.bfloat16, 1005, 1)
    a, g = syn.uclip_params(1536, False, True, 1005)
    y = torch.empty_like(x)
    timed("dyht", 2 * 512 * 1536 * 2, "512 x 1536", lambda: oracle.dyht(x, a, g, y))
    B, ctx = 4, 1024
    q, cache, table, seq = syn.attention_inputs(B, ctx, 12, 2, 128, 16, 4096, torch.bfloat16, 1012)
    o = torch.empty_like(q)
    timed("decode_attention", 2 * B * ctx * 2 * 128 * 2, f"B={B} x {ctx} tokens",
          lambda: oracle.paged_decode_attention(q, cache, table, seq, o))
    out["decode_attention_ws"] = out["decode_attention"]  # same result; the workspace only splits the work
    K, N = syn.QWEN25_QKV["K"], syn.QWEN25_QKV["N"]
    x = syn.normal((1, K), 0.0, 1.0, torch.bfloat16, 1030, 1)
    w = syn.normal((K,), 1.0, 0.1, torch.bfloat16, 1030, 2)
    W = syn.linear_weight(N, K, torch.bfloat16, 1030)
    y = torch.empty(1, N, dtype=torch.bfloat16)
    timed("rmsnorm_linear", N * K * 2, "B=1", lambda: oracle.rmsnorm_linear(x, w, W, y, syn.EPS))
    I, N = syn.QWEN25_DOWN["I"], syn.QWEN25_DOWN["N"]
    gu = syn.normal((1, 2 * I), 0.0, 1.0, torch.bfloat16, 1031, 3)
    W = syn.linear_weight(N, I, torch.bfloat16, 1031)
    y = torch.empty(1, N, dtype=torch.bfloat16)
    timed("swiglu_linear", N * I * 2, "B=1", lambda: oracle.glu_linear(gu, W, y, "silu"))
    # the workspace entry points compute the same result
    out["rmsnorm_linear_ws"] = out["rmsnorm_linear"]
    out["swiglu_linear_ws"] = out["swiglu_linear"]
    return out


# --------------------------------------------------------------------------- main (GPU)
def order_entries(entries):
    """Step order: the largest streams first (SwiGLU T=4096, the dominant kernel, opens the step
    right after the L2 clean-up), then GLU, add_rmsnorm, RoPE, the RMSNorm sweep, the chains."""
    rank = {"swiglu": 0, "reglu": 0, "add_rmsnorm": 1, "rope_kv_store": 2, "rmsnorm": 3, "chain": 4,
            "uclip": 5, "decode_attention": 6, "linear": 7}
    return sorted(entries, key=lambda e: (rank[e.op], -e.bytes, e.op != "swiglu", e.name))


def run_gpu(args):
    import torch

    import swiglu_rmsnorm_add_gb300 as sra

    rank, world, local = dist_setup(args)
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.current_stream(dev)
    sh = int(stream.cuda_stream)
    only = [o for o in args.only.split(",") if o]
    pdl = not args.no_pdl
    sra.set_pdl(pdl)
    for f in (x for x in args.force.split(",") if x):
        op, v = f.split("=")
        sra.force_variant(op, int(v, 0))

    entries = build_entries(dev, sh, only)
    if only:  # a companion shape named on the command line is timed as a step entry of its own
        entries += build_entries(dev, sh, only, companions=True)
    entries = order_entries(entries)
    if not args.no_chain and (not only or any(o.startswith("chain") for o in only)):
        for B in (1, 64):
            entries.append(ChainEntry(B, dev, pdl))
    assert entries, "nothing selected"
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    bytes_per_step = sum(e.bytes for e in entries)
    launches_per_step = sum(112 if e.op == "chain" else 1 for e in entries)
    kern = [i for i, e in enumerate(entries) if e.op != "chain"] or list(range(len(entries)))
    dom = max(kern, key=lambda i: (entries[i].bytes, entries[i].op == "swiglu"))

    def clean_l2():
        # write a buffer larger than L2 (evicts everything), then read it back so
        # the lines left in L2 are clean and no write-back lands in the timed step
        flush.fill_(1)
        flush.sum()

    def enqueue_step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        for i, e in enumerate(entries):
            if ev is not None and i == dom:
                ev[1].record(stream)
            e.launch()
            if ev is not None and i == dom:
                ev[2].record(stream)
        if ev is not None:
            ev[3].record(stream)

    # host enqueue time of one step -> a device-side delay that keeps the GPU behind the host
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    t0 = time.perf_counter()
    enqueue_step(evs)
    host_s = time.perf_counter() - t0
    torch.cuda.synchronize()
    delay_cycles = int(min(2e7, max(2e5, 3.0 * host_s * 2.0e9)))

    def step(ev=None):
        clean_l2()
        torch.cuda._sleep(delay_cycles)
        if ev is not None:
            torch.cuda.nvtx.range_push(NVTX_STEP)  # lets ncu --nvtx-include select the timed steps
        enqueue_step(ev)
        if ev is not None:
            torch.cuda.nvtx.range_pop()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(local)
    clocks = ClockSampler(gpu_id)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    for k in range(args.steps):
        step(ev[k])
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - w0
    time.sleep(0.25)
    clk = clocks.stop()

    step_ms = [ev[k][0].elapsed_time(ev[k][3]) for k in range(args.steps)]
    dom_ms = [ev[k][1].elapsed_time(ev[k][2]) for k in range(args.steps)]
    ms = reduce_max(statistics.fmean(step_ms), dev)
    value = weak_value(bytes_per_step, ms, world)

    peak, peak_src = measured_peak()
    de = entries[dom]
    d_us = statistics.fmean(dom_ms) * 1e3
    achieved = de.bytes / (d_us * 1e-6) / 1e9
    traffic = kernel_traffic(de.name)
    roofline = {"bound": "hbm", "kernel": de.name, "achieved": round(achieved, 1), "peak": peak,
                "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": traffic, "algorithmic_bytes": de.bytes,
                "us_per_launch": round(d_us, 3), "timed": "CUDA events around its launch in every timed step"}
    if traffic:
        # the same launch on the DRAM bytes ncu counts for one launch: writes still dirty in L2 when
        # the launch ends are written back later, so this is the rate the launch itself sustained
        roofline["achieved_on_traffic"] = round(traffic / (d_us * 1e-6) / 1e9, 1)
        roofline["frac_on_traffic"] = round(traffic / (d_us * 1e-6) / 1e9 / peak, 4)

    # per-kernel table: each launch timed alone (clean L2, event pair), after the step loop
    reps = max(10, min(50, args.steps))

    def time_alone(fn, n):
        out = []
        for _ in range(n):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            clean_l2()
            torch.cuda._sleep(200000)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            out.append(a.elapsed_time(b))
        return out

    cap_stream = torch.cuda.Stream(dev)

    def graph_of(calls):
        """The calls (launched on cap_stream) captured into one CUDA graph, so a replay
        measures the device alone: the host's enqueue rate cannot pace the launches."""
        with torch.cuda.stream(cap_stream):
            for c in calls:
                c()
        cap_stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap_stream):
            for c in calls:
                c()
        return g

    def time_stream(e):
        """Per-launch time of back-to-back launches, each on its own copy of the
        buffers (the copies together exceed 4x L2, so every launch reads cold data),
        replayed from a CUDA graph."""
        n = int(min(64, max(1, -(-STREAM_BYTES // max(1, e.bytes)))))
        calls = e.replicas(n, int(cap_stream.cuda_stream))
        g = graph_of(calls)
        rounds = max(2, 8 // len(calls)) if len(calls) < 8 else 3
        per = []
        for _ in range(rounds):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            clean_l2()
            torch.cuda._sleep(200000)
            a.record(stream)
            g.replay()
            b.record(stream)
            b.synchronize()
            per.append(a.elapsed_time(b) / len(calls))
        del g, calls
        return statistics.median(per), n

    per_kernel = []
    for e in entries:
        times = time_alone(e.launch, reps)
        us = statistics.fmean(times) * 1e3
        srt = sorted(times)
        rec = {"name": e.name, "bytes": e.bytes, "us_alone": round(us, 3),
               "us_alone_p20": round(srt[len(srt) // 5] * 1e3, 3),
               "us_alone_p80": round(srt[(4 * len(srt)) // 5] * 1e3, 3)}
        if e.op != "chain":
            st_ms, copies = time_stream(e)
            su = st_ms * 1e3
            rec.update({"us": round(su, 3), "copies": copies, "gbs": round(e.bytes / (su * 1e-6) / 1e9, 1),
                        "frac_of_peak": round(e.bytes / (su * 1e-6) / 1e9 / peak, 4),
                        "rows_per_s": round(e.rows / (su * 1e-6), 1)})
        else:
            rec.update({"us": round(us, 3), "gbs": round(e.bytes / (us * 1e-6) / 1e9, 1),
                        "frac_of_peak": round(e.bytes / (us * 1e-6) / 1e9 / peak, 4),
                        "rows_per_s": round(e.rows / (us * 1e-6), 1)})
        if e.op == "chain":
            rec["tokens_per_s"] = rec.pop("rows_per_s")
            rec["launches"] = 112
            rec["us_per_launch"] = round(us / 112, 3)
            rec["pdl"] = pdl
            # A/B: the same chain captured without programmatic dependent launch
            g_main = e.chain.graph
            e.chain.capture(pdl=not pdl, warmup=False)
            t_alt = time_alone(e.chain.replay, reps)
            e.chain.graph = g_main
            rec["us_other_pdl_setting"] = round(statistics.fmean(t_alt) * 1e3, 3)
            # A/B: the same step launched eagerly from the host (112 C-ABI calls through the binding)
            t_eager = time_alone(e.chain.step, max(5, reps // 4))
            rec["us_eager"] = round(statistics.fmean(t_eager) * 1e3, 3)
            # per kernel kind inside the chain: a graph of only that kind's launches, in chain order
            # on the chain's buffers (each launch waits for the one before, as in the step)
            kinds = {}
            nl = e.chain.launches_per_step()
            for kind, kb in e.bytes_by_kind.items():
                gk = e.chain.capture_kind(kind, pdl)
                tk = statistics.fmean(time_alone(gk.replay, reps)) * 1e3
                del gk
                kinds[kind] = {"launches": nl[kind], "bytes": kb, "us": round(tk, 3),
                               "us_per_launch": round(tk / nl[kind], 3),
                               "gbs": round(kb / (tk * 1e-6) / 1e9, 1),
                               "frac_of_peak": round(kb / (tk * 1e-6) / 1e9 / peak, 4)}
            rec["kinds"] = kinds
            rec["kinds_what"] = ("each kernel kind of the step alone: a CUDA graph of its launches in chain order "
                                 "on the chain's own buffers, replayed (clean L2 before each replay)")
        per_kernel.append(rec)

    # launch latency: back-to-back launches of a one-row RMSNorm (1 x 128 bf16),
    # queued behind a device delay so the host is ahead; with and without PDL
    latency = {}
    if not only:
        from swiglu_rmsnorm_add_gb300 import synthetic as syn

        xt, wt = syn.rms_inputs(1, 128, torch.bfloat16, 7)
        xt, wt = xt.to(dev), wt.to(dev)
        ot = torch.empty_like(xt)
        L = sra.lib()
        targs = (xt.data_ptr(), wt.data_ptr(), ot.data_ptr(), 1, 128, 128, 128, 1e-6, 2,
                 int(cap_stream.cuda_stream))
        for mode in (True, False):
            prev = sra.set_pdl(mode)
            n = 200
            g = graph_of([lambda: L.sra_rmsnorm(*targs)] * n)
            per = []
            for _ in range(3):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda._sleep(200000)
                a.record(stream)
                g.replay()
                b.record(stream)
                b.synchronize()
                per.append(a.elapsed_time(b) * 1e3 / n)
            sra.set_pdl(prev)
            del g
            latency["pdl" if mode else "no_pdl"] = round(statistics.median(per), 3)
        latency["what"] = ("us per launch, 200 back-to-back rmsnorm [1,128] bf16 launches replayed from a CUDA graph "
                           "(the per-launch floor of a dependent kernel chain)")
        # per kernel: the time the launch could take at best in such a chain (its bytes at the
        # measured copy bandwidth plus that per-launch floor), and the fraction of it reached
        if pdl:
            for rec in per_kernel:
                if "frac_of_peak" in rec and not rec["name"].startswith("chain"):
                    floor = rec["bytes"] / peak / 1e3 + latency["pdl"]
                    rec["floor_us"] = round(floor, 3)
                    rec["frac_of_floor"] = round(floor / rec["us"], 4)

    # companions (row-scaled shapes, >= 256 MB traffic), timed alone
    companions = []
    if not args.no_companions and not only:
        comp = build_entries(dev, sh, companions=True)
        for e in comp:
            for _ in range(3):
                e.launch()
            times = time_alone(e.launch, reps)
            ua = statistics.fmean(times) * 1e3
            st_ms, copies = time_stream(e)
            us = st_ms * 1e3
            companions.append({"name": e.name, "bytes": e.bytes, "us_alone": round(ua, 2), "us": round(us, 2),
                               "copies": copies, "gbs": round(e.bytes / (us * 1e-6) / 1e9, 1),
                               "frac_of_peak": round(e.bytes / (us * 1e-6) / 1e9 / peak, 4)})
        del comp

    # end to end through the C ABI from pinned host buffers
    e2e = None
    if not args.no_e2e:
        # per launch: the inputs it is the first to read (host -> device) and its outputs
        # (device -> host). The copies run on two copy streams beside the launches' stream,
        # so the two directions overlap each other and the kernels: a launch waits for its
        # own inputs only, its outputs leave as soon as it is done, and a launch that
        # rewrites a buffer an earlier launch's read-back still reads waits for that read.
        # (No launch of the step writes a buffer another launch reads, so an input may be
        # copied in while earlier launches run.)
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        plan = []
        seen = set()
        for e in entries:
            ins = []
            for t in e.inputs:
                if t.data_ptr() not in seen:
                    seen.add(t.data_ptr())
                    ins.append((torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu()), t))
            outs = [(t, torch.empty(t.shape, dtype=t.dtype, pin_memory=True)) for t in e.outputs]
            plan.append((e, ins, outs))
        h2d = sum(h.numel() * h.element_size() for _, ins, _ in plan for h, _ in ins)
        d2h = sum(h.numel() * h.element_size() for _, _, outs in plan for _, h in outs)

        def e2e_step():
            reading = {}  # device buffer -> event after its latest read-back
            for e, ins, outs in plan:
                if ins:
                    with torch.cuda.stream(s_in):
                        for h, d in ins:
                            d.copy_(h, non_blocking=True)
                    stream.wait_stream(s_in)
                for d, _ in outs:
                    ev = reading.get(d.data_ptr())
                    if ev is not None:
                        stream.wait_event(ev)
                e.launch()
                if outs:
                    s_out.wait_stream(stream)
                    with torch.cuda.stream(s_out):
                        for d, h in outs:
                            h.copy_(d, non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(s_out)
                    for d, _ in outs:
                        reading[d.data_ptr()] = ev
            stream.wait_stream(s_out)
            stream.synchronize()

        for _ in range(max(2, args.warmup)):
            e2e_step()
        n_e2e = max(5, min(args.steps, 50))
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        if world > 1:
            dist.barrier()
        e_s = reduce_max((time.perf_counter() - t0) / n_e2e, dev)
        e2e = {"value": round(weak_value(bytes_per_step, e_s * 1e3, world), 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(e_s * 1e3, 3),
               "how": "host wall time per step; pinned-host inputs in and outputs out on two copy streams that "
                      "overlap each other and the launches (each launch waits for its own inputs)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu and not only:
        cpu = cpu_sample_run(args.cpu_seconds)
        cpu = {k: (round(v, 4) if isinstance(v, float) else v) for k, v in cpu.items()}
        if companions:
            # the oracle beside each widened row: one thread on a small sample of the row's workload
            rows_cpu = cpu_rows_run()
            for c in companions:
                for prefix, r in rows_cpu.items():
                    if c["name"].startswith(prefix + ":"):
                        c["cpu_oracle_gbs"] = r["gbs"]
                        c["cpu_oracle_sample"] = f"{r['sample']}, 1 thread, {r['seconds']} s"
            cpu["rows"] = rows_cpu

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded host RNG, resident in HBM)",
                "config": {"workload": WORKLOAD if not only else f"subset: {','.join(only)}",
                           "io_dtypes": "bf16 (rmsnorm sweep also fp32, fp16); arithmetic fp32",
                           "l2": "flushed before every step: a 256 MiB device write, then a read of it",
                           "bytes_per_step": bytes_per_step, "launches_per_step": launches_per_step,
                           "programmatic_dependent_launch": pdl,
                           "parallelism": f"replicas x{world} (no collective)",
                           "step_wall_ms_incl_flush_and_delay": round(wall / args.steps * 1e3, 3)},
                "gpu_launches": launches_per_step * args.steps,
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
                "launch_latency_us": latency, "kernels": per_kernel, "companions": companions}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_sweep(args):
    """Streaming time of every RMSNorm variant on every norm shape, and of every GLU
    variant on the GLU shapes (dispatch evidence); projection and decode-attention
    variants on the companion shapes named with --only."""
    import torch

    import swiglu_rmsnorm_add_gb300 as sra

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    sh = int(stream.cuda_stream)
    sra.set_pdl(not args.no_pdl)
    swept = ("rmsnorm", "add_rmsnorm", "swiglu", "reglu", "linear", "decode_attention")
    only = [o for o in args.only.split(",") if o] or list(swept[:4])
    entries = [e for e in build_entries(dev, sh, only) if e.op in swept]
    if not args.only:
        entries += [e for e in build_entries(dev, sh, companions=True) if e.op in swept[:4]]
    else:  # companion shapes named on the command line
        entries += [e for e in build_entries(dev, sh, only, companions=True) if e.op in swept]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    peak, _ = measured_peak()
    table = []
    for e in entries:
        row = {"name": e.name, "bytes": e.bytes, "auto": None, "variants": {}}
        n = int(min(64, max(1, -(-STREAM_BYTES // max(1, e.bytes)))))
        calls = e.replicas(n) if n > 1 else [e.launch]
        op = {"swiglu": "glu", "reglu": "glu", "linear": "linear",
              "decode_attention": "decode_attention"}.get(e.op, "rmsnorm")
        settings = [(-1, "auto")]
        for v in range(sra.variant_count(op)):
            nm = sra.variant_name(op, v)
            if nm in ("warp_rows", "cta_row", "cta_pair", "cta_lean"):
                nvs = (1, 2, 3, 4, 6, 8, 12, 16) if nm == "warp_rows" else (1, 2, 3, 4, 6, 8)
                settings += [(v | (nv << 8), f"{nm}/nv{nv}") for nv in nvs]
            elif nm == "tcgen05":
                settings += [(v, nm)] + [(v | (sk << 8) | (st << 16), f"{nm}/splits{sk}/stages{st}")
                                         for st in (4, 8) for sk in (4, 6, 8, 10, 12, 16)]
            elif op == "decode_attention" and nm != "cuda_cores":
                settings += [(v, nm)] + [(v | (sk << 8), f"{nm}/splits{sk}") for sk in (1, 2, 4, 8, 16)]
                if nm == "mma_sync":   # 4-warp CTAs, two per SM
                    settings += [(v | (4 << 16) | (sk << 8), f"{nm}/w4" + (f"/splits{sk}" if sk else ""))
                                 for sk in (0, 1, 2, 4, 8, 16)]
            elif nm == "warps_row":
                settings += [(v | (nv << 8) | (g << 16), f"{nm}/g{g}nv{nv}") for g in (2, 4, 8) for nv in (8, 16)]
            else:
                settings.append((v, nm))
        if op == "rmsnorm" and args.sweep_cps:
            # the same register variants with at most c CTAs per SM (grid = c x SMs)
            base = [(1, "cta_row", nv, 0) for nv in (2, 4, 8)] + [(7, "cta_lean", nv, 0) for nv in (4, 8)]
            base += [(8, "warps_row", 16, 4), (8, "warps_row", 8, 8)]
            for v, nm, nv, g in base:
                for c in (1, 2, 3, 4, 6):
                    settings.append((v | (nv << 8) | (g << 16) | (c << 24), f"{nm}/nv{nv}" + (f"g{g}" if g else "")
                                     + f"/cps{c}"))
        for v, label in settings:
            sra.force_variant(op, v)
            try:
                for c in calls:
                    c()
            except RuntimeError:
                continue
            per = []
            # an NVTX range per (shape, setting): an ncu launch list of this sweep can be split by it
            torch.cuda.nvtx.range_push(f"sweep:{e.name}|{label}")
            for _ in range(3):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                flush.fill_(1)
                flush.sum()
                torch.cuda._sleep(200000)
                a.record(stream)
                for c in calls:
                    c()
                b.record(stream)
                b.synchronize()
                per.append(a.elapsed_time(b) * 1e3 / len(calls))
            torch.cuda.nvtx.range_pop()
            us = statistics.median(per)
            rec = {"us": round(us, 3), "frac": round(e.bytes / (us * 1e-6) / 1e9 / peak, 4)}
            if v < 0:
                row["auto"] = rec
            else:
                row["variants"][label] = rec
        sra.force_variant(op, -1)
        del calls
        table.append(row)
    print(json.dumps({"variant_sweep": table, "peak_gbs": peak, "timing": "back-to-back launches over rotating "
                      "copies (>= 512 MiB), median of 3, us per launch"}), flush=True)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    # warm-up samples, then K timed samples of the oracle over a bounded fraction of the step
    frac = None
    vals = []
    res = None
    for i in range(args.warmup + args.steps):
        res = cpu_sample_run(args.cpu_seconds / max(1, args.steps), fraction=frac)
        frac = res["fraction"]
        if i >= args.warmup:
            vals.append(res)
    secs = sum(r["seconds"] for r in vals)
    b = sum(r["bytes"] for r in vals)
    value = b / secs / 1e9
    cpu = {"value": round(value, 4), "unit": UNIT, "cores": res["cores"], "kind": "oracle", "sample": res["sample"]}
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(secs / len(vals) * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded host RNG)",
            "config": {"workload": WORKLOAD, "sample_fraction": frac},
            "cpu_baseline": cpu, "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                                         "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    elif a.sweep_variants:
        run_sweep(a)
    else:
        run_gpu(a)
