#!/usr/bin/env python
"""GPTQ per-layer quantization benchmark on GB300.

One step = one whole layer pass of the workload: Hessian accumulate + finalize,
prepare (dead fix, damping, act_order, U), and the GPTQ column loop + packing for
every weight that shares the layer input. Inputs are seeded synthetic layers.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl ours|reference]
  python bench.py --op dequant_matmul [--config C] [--tokens T]   (the stored-form consumer)
  python bench.py --op layerwise [--mlp mlp4096|toy]             (apply_layerwise on a synthetic MLP)
  python bench.py --op quantize [--shape 4096x14336] [--bits B]   (the column loop alone)

Prints one JSON line. `value` is milliseconds per layer pass (lower is better),
device-timed with CUDA events, L2 flushed between steps when the inputs fit in it.
`e2e` is the same pass through the C ABI from pinned host buffers, host<->device
copies included. `roofline` is for the kernel with the largest share of the step,
from a second, profiled pass over the same steps. `cpu_baseline` times the CPU
oracle on this host (test infrastructure, reported for context).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GPTQ layer quantize time (ms, incl. H+Cholesky) and % of roofline per kernel"
L2_BYTES = 129 * 1024 * 1024
FFMA_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12   # SMs x FP32 lanes x 2 flop x max SM clock
# the Llama-3-8B-shaped decoder block (7 linears x bits 2, 3, 4 on 262144 calibration tokens)
DEFAULT_CONFIG = 4


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-profile", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time eager steps instead of CUDA-graph replays")
    ap.add_argument("--op", choices=["layer", "dequant_matmul", "layerwise", "quantize"], default="layer")
    ap.add_argument("--shape", default="4096x14336", help="rows x cols of --op quantize's weight stack")
    ap.add_argument("--mlp", default="mlp4096")
    ap.add_argument("--tokens", type=int, default=8192)
    # smaller cases of the same shapes (profiler captures that must stay within a few GB):
    # fewer calibration tokens per layer input, or one bit width of the decoder block's sweep
    ap.add_argument("--x-tokens", type=int, default=0, help="calibration tokens per input (default: the workload's)")
    ap.add_argument("--bits", type=int, default=0, help="keep only the layers of this bit width")
    # the timed step's schedule: serial (group after group), prepare (all Hessians, then the
    # groups' gptq_prepare calls side by side, then the quantizations), groups (all
    # Hessians, then each group's prepare and quantizations on its own stream), layers (as
    # groups, with each layer of a group quantised on a stream of its own)
    ap.add_argument("--schedule", choices=["serial", "prepare", "groups", "layers"], default="layers")
    return ap.parse_args(argv)


def workload_for(args):
    """The workload recipe, reduced by --x-tokens / --bits when given (the name says so)."""
    import dataclasses
    import synth
    wl = synth.workload(args.config)
    if not args.x_tokens and not args.bits:
        return wl
    layers = [L for L in wl.layers if not args.bits or L.q.bits == args.bits]
    if not layers:
        raise SystemExit(f"no layer of {args.bits} bits in workload {args.config}")
    if args.x_tokens:
        layers = [dataclasses.replace(L, x=dataclasses.replace(L.x, n=args.x_tokens)) for L in layers]
    name = wl.name + (f"-x{args.x_tokens}" if args.x_tokens else "") + (f"-only{args.bits}b" if args.bits else "")
    return dataclasses.replace(wl, name=name, layers=layers)


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ----------------------------------------------------------------------------- clocks

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            # wait (at most 3 s) for the first sample, so that a short timed region that
            # follows is still bracketed by samples
            t0 = time.perf_counter()
            while time.perf_counter() - t0 < 3.0 and os.path.getsize(self.path) == 0:
                time.sleep(0.02)
        except Exception:  # noqa: BLE001
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:  # noqa: BLE001
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- workload

class Layer:
    """One layer input X and the weights that read it. The weights live stacked by rows in
    one (sum of rows, cols) matrix `Wcat` (a fused projection); `Ws` are its row blocks.
    GPTQ's rows are independent given U, so one gptq_quantize over Wcat equals one call per
    weight, row for row."""

    def __init__(self, spec, X, Wcat, Ws, names):
        self.spec = spec
        self.X = X
        self.Wcat = Wcat
        self.Ws = Ws
        self.names = names


def x_group(cfg: int, wl, li: int) -> int:
    """Which distinct input layer li of the workload reads: the decoder block's four inputs
    (q/k/v, o, gate/up, down) repeat across its bit widths; elsewhere one input per layer."""
    if cfg != 4:
        return li
    return ("q_proj", "o_proj", "gate_proj", "down_proj").index(wl.layers[li].weights[0].name)


def build_layers(cfg: int, device, host: bool = False, wl=None):
    import torch
    import synth
    wl = wl or synth.workload(cfg)
    layers = []
    xcache = {}
    for li, L in enumerate(wl.layers):
        key = (L.x, x_group(cfg, wl, li))
        if key not in xcache:
            seed = synth.x_seed(cfg, L.x) + (key[1] if cfg == 4 else 0)
            xcache[key] = synth.make_x(L.x, seed, device=device)
        X = xcache[key]
        cols = L.weights[0].inp
        Wcat = torch.empty(sum(w.out for w in L.weights), cols, dtype=torch.float32, device=device)
        Ws, r0 = [], 0
        for w in L.weights:
            Wcat[r0:r0 + w.out].copy_(synth.make_weight(w.out, w.inp, w.std, synth.weight_seed(cfg, w.name),
                                                        device=device))
            Ws.append(Wcat[r0:r0 + w.out])
            r0 += w.out
        layers.append(Layer(L, X, Wcat, Ws, [w.name for w in L.weights]))
    return wl, layers


class Runner:
    """Holds preallocated outputs/workspaces so a step only enqueues library calls: per
    layer one Hessian pass, one gptq_prepare and one gptq_quantize over the stacked weights."""

    def __init__(self, lib, layers, device):
        import torch
        self.lib = lib
        self.layers = layers
        self.dev = device
        self.hess = {}
        self.prep_ws = {}
        self.q_ws = {}
        self.outs = []
        # layers that read the same X with the same damping and ordering share H, U, perm
        # and dead: one Hessian pass and one gptq_prepare per group (the bit-width sweep of
        # a decoder block re-quantises the same inputs)
        self.groups = []
        gkey = {}
        for li, L in enumerate(layers):
            key = (id(L.X), L.spec.q.damp, L.spec.q.act_order)
            if key not in gkey:
                gkey[key] = len(self.groups)
                self.groups.append([])
            self.groups[gkey[key]].append(li)
        for L in layers:
            d = L.X.shape[1]
            if d not in self.hess:
                self.hess[d] = lib.Hessian(d, device)
            q = L.spec.q
            r, c = L.Wcat.shape
            G = -(-c // q.group) if q.group else 1
            self.outs.append({
                "codes": torch.empty(r, c, dtype=torch.int8, device=device),
                "scales": torch.empty(r, G, dtype=torch.float32, device=device),
                "zeros": torch.empty(r, G, dtype=torch.uint8, device=device),
                "g_idx": torch.empty(c, dtype=torch.int32, device=device),
                "Wq": torch.empty(r, c, dtype=torch.float32, device=device),
                "packed": torch.empty(r, lib.gptq_packed_words_per_row(c, q.bits), dtype=torch.int32,
                                      device=device),
                "row_loss": torch.empty(r, dtype=torch.float32, device=device),
            })

        # one prepare workspace and one quantize workspace per group (the concurrent schedule
        # runs groups side by side; a group's calls share them in turn), and one stream per
        # group for it
        for g in self.groups:
            d = layers[g[0]].X.shape[1]
            self.prep_ws[id(g)] = torch.empty(lib.gptq_prepare_workspace_bytes(d, True), dtype=torch.uint8,
                                              device=device)
            nb = 0
            for li in g:
                q = layers[li].spec.q
                r, c = layers[li].Wcat.shape
                nb = max(nb, lib.gptq_quantize_workspace_bytes(r, c, q.bits, q.group, q.sym))
            self.q_ws[id(g)] = torch.empty(nb, dtype=torch.uint8, device=device)
        self.gstreams = [torch.cuda.Stream(device=device) for _ in self.groups]
        # per layer (made on first use by the layers schedule): a stream and a quantize
        # workspace, so the layers of a group (the bit widths of one input) quantise side by side
        self.lstreams = {}
        self.q_ws_layer = {}

    def _layer_res(self, li):
        import torch
        if li not in self.lstreams:
            L = self.layers[li]
            q = L.spec.q
            r, c = L.Wcat.shape
            self.q_ws_layer[li] = torch.empty(self.lib.gptq_quantize_workspace_bytes(r, c, q.bits, q.group, q.sym),
                                              dtype=torch.uint8, device=self.dev)
            self.lstreams[li] = torch.cuda.Stream(device=self.dev)
        return self.lstreams[li], self.q_ws_layer[li]

    def step_concurrent(self, quantize_in_group: bool = True, Xs=None, Wcats=None, x_chunks=None, w_ready=None,
                        layer_done=None, order=None, fork_layers: bool = False):
        """One pass with the groups side by side: every group's Hessian on the current stream
        (each is a full-GPU kernel), then per group on its own stream, as soon as that group's
        Hessian is final (an event, not the whole Hessian queue), its gptq_prepare - the
        small groups' latency-bound factorisations overlap the large group's - followed, with
        quantize_in_group, by its gptq_quantize calls (else those run after all prepares, on
        the current stream). With fork_layers each layer of a group then quantises on a
        stream and workspace of its own, forked from the group's stream after its prepare.
        The same calls and results as step(); Xs, Wcats, x_chunks, w_ready, layer_done and
        order as there."""
        import torch
        lib = self.lib
        main = torch.cuda.current_stream()
        order = list(order) if order is not None else list(range(len(self.groups)))
        Hs = {}
        for gi in order:
            g = self.groups[gi]
            X = self.layers[g[0]].X if Xs is None else Xs[g[0]]
            h = self.hess[X.shape[1]]
            h.reset()
            if x_chunks is None:
                h.accumulate(X)
            else:
                for rows, ev, _ in x_chunks[gi]:
                    main.wait_event(ev)
                    h.accumulate(rows)
            Hs[gi] = h.finalize()[:2]
            ev = torch.cuda.Event()
            ev.record(main)
            Hs[gi] = (Hs[gi], ev)
        preps = {}
        for gi in order:
            g = self.groups[gi]
            st = self.gstreams[gi]
            (H, diag), ev = Hs[gi]
            st.wait_event(ev)
            with torch.cuda.stream(st):
                q0 = self.layers[g[0]].spec.q
                U, perm, dead = lib.gptq_prepare(H, diag, q0.damp, act_order=q0.act_order, ws=self.prep_ws[id(g)])
                preps[gi] = (U, perm, dead)
                if quantize_in_group:
                    self._quantize_group(g, U, perm, dead, Wcats, w_ready, layer_done, fork_layers)
        for st in self.gstreams:
            main.wait_stream(st)
        if not quantize_in_group:
            for gi in order:
                self._quantize_group(self.groups[gi], *preps[gi], Wcats, w_ready, layer_done)
        return self.outs

    def _quantize_group(self, g, U, perm, dead, Wcats=None, w_ready=None, layer_done=None, fork_layers=False):
        import torch
        gst = torch.cuda.current_stream()
        for li in g:
            L = self.layers[li]
            Wcat = L.Wcat if Wcats is None else Wcats[li]
            q = L.spec.q
            st, ws = (self._layer_res(li) if fork_layers else (gst, self.q_ws[id(g)]))
            if st is not gst:
                st.wait_stream(gst)
            with torch.cuda.stream(st):
                if w_ready is not None:
                    st.wait_event(w_ready[li])
                self.lib.gptq_quantize(Wcat, U, perm, dead, q.bits, q.group, q.sym, ws=ws, out=self.outs[li])
                if layer_done is not None:
                    layer_done[li].record(st)
        if fork_layers:
            for li in g:
                gst.wait_stream(self.lstreams[li])

    def weight_outputs(self, li):
        """The outputs of layer li split per weight (row blocks of the stacked outputs)."""
        o, res, r0 = self.outs[li], [], 0
        for W in self.layers[li].Ws:
            r1 = r0 + W.shape[0]
            res.append({k: (v if k == "g_idx" else v[r0:r1]) for k, v in o.items()})
            r0 = r1
        return res

    def step(self, events=None, Xs=None, Wcats=None, x_chunks=None, w_ready=None, layer_done=None, order=None):
        """One pass over every layer: per group one Hessian pass and one gptq_prepare, then
        one gptq_quantize per layer; `events` collects (start, H done, U done, end) CUDA
        events per group, followed by (layer, event after its quantisation) per layer. For inputs copied in on another stream: the Hessian of group g
        accumulates x_chunks[g] = [(token rows of its input, event, first row), ...] chunk by chunk,
        each once its copy has landed; the step waits for w_ready[li] (layer li's weights)
        just before it uses them, and records layer_done[li] once layer li's outputs are
        written. `order` is the order of the groups (default: as listed)."""
        import torch
        lib = self.lib
        for gi in (order if order is not None else range(len(self.groups))):
            g = self.groups[gi]
            L0 = self.layers[g[0]]
            X = L0.X if Xs is None else Xs[g[0]]
            q0 = L0.spec.q
            h = self.hess[X.shape[1]]
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)] if events is not None else None
            if e:
                e[0].record()
            h.reset()
            if x_chunks is None:
                h.accumulate(X)
            else:
                for rows, ev, _ in x_chunks[gi]:
                    torch.cuda.current_stream().wait_event(ev)
                    h.accumulate(rows)
            H, diag, _ = h.finalize()
            if e:
                e[1].record()
            U, perm, dead = lib.gptq_prepare(H, diag, q0.damp, act_order=q0.act_order, ws=self.prep_ws[id(g)])
            if e:
                e[2].record()
            for li in g:
                L = self.layers[li]
                Wcat = L.Wcat if Wcats is None else Wcats[li]
                q = L.spec.q
                if w_ready is not None:
                    torch.cuda.current_stream().wait_event(w_ready[li])
                lib.gptq_quantize(Wcat, U, perm, dead, q.bits, q.group, q.sym, ws=self.q_ws[id(g)],
                                  out=self.outs[li])
                if layer_done is not None:
                    layer_done[li].record()
                if e:   # after each layer's quantisation: (layer, event)
                    le = torch.cuda.Event(enable_timing=True)
                    le.record()
                    e.append((li, le))
            if e:
                e[3].record()
                events.append(e)
        return self.outs


def flush_l2(buf):
    buf.zero_()


def stage_breakdown(evs, groups, layers, steps: int):
    """Per input group and per bit width from the events of serial steps (Runner.step's
    `events`: per group and step, (start, H done, U done, end) then (layer, event after
    its quantisation) per layer; the groups in order within each step). Per group: H and
    U once, then each layer's quantisation; per bit width: its quantisations summed,
    "fresh" (the H and U of its inputs counted again for it) and "amortised" (H and U
    shared over the layers that read the same inputs). Milliseconds per step."""
    ng = len(groups)
    per_group, by_bits = [], {}
    for gi, g in enumerate(groups):
        es = evs[gi::ng]
        hp = [sum(e[a].elapsed_time(e[b]) for e in es) / steps for a, b in ((0, 1), (1, 2))]
        qs = {}
        for e in es:
            prev = e[2]
            for li, le in e[4:]:
                qs[li] = qs.get(li, 0.0) + prev.elapsed_time(le) / steps
                prev = le
        per_group.append({"input": list(layers[g[0]].X.shape), "layers": [layers[li].names for li in g],
                          "hessian": hp[0], "prepare": hp[1],
                          "quantize": {str(layers[li].spec.q.bits) + "b " + "+".join(layers[li].names): qs[li]
                                       for li in g}})
        for bits in sorted({layers[li].spec.q.bits for li in g}):
            mine = [li for li in g if layers[li].spec.q.bits == bits]
            b = by_bits.setdefault(bits, {"quantize": 0.0, "fresh": 0.0, "amortised": 0.0})
            qb = sum(qs[li] for li in mine)
            b["quantize"] += qb
            b["fresh"] += qb + hp[0] + hp[1]
            b["amortised"] += qb + (hp[0] + hp[1]) * len(mine) / len(g)
    return per_group, {str(k): v for k, v in sorted(by_bits.items())}


def algorithmic(cfg_layers):
    """Per-kernel-class algorithmic work for one step: fp32/bf16 FLOPs, or bytes for the
    memory-bound kernels (the unit is fixed per class in ROOF)."""
    work = {}

    def add(k, v):
        work[k] = work.get(k, 0.0) + v

    NB, QB = 128, 128
    seen = set()
    for L in cfg_layers:
        n, d = L.X.shape
        key = (id(L.X), L.spec.q.damp, L.spec.q.act_order)
        first = key not in seen    # H and U once per shared input (as Runner does)
        seen.add(key)
        if first:
            add("hessian_tc_kernel", 2.0 * n * d * (d + 1) / 2)
        # prepare: per 128-wide panel, potrf (Cholesky n^3/3 + inverse n^3/6 FMA), the panel
        # solve 2 m n^2, the lower SYRK 2 m(m+1)/2 n, the inverse's scale 2 n k n and
        # trailing update 2 m k n (k = columns filled so far)
        # The factorisation's critical chain (class [chain]) computes per panel its solve
        # and the rank update of the next panel's columns (lower part), with this panel's
        # L21 inside a super-panel and with all its panels' at the super-panel's end; the
        # rest of the same work is the side stream's (class [prepare]). The two add up to
        # the total above: every product is computed once, by one of them.
        spw = 4 * NB if d >= 2048 else NB
        for k0 in (range(0, d, NB) if first else ()):
            nb = min(NB, d - k0)
            m = d - k0 - nb
            ncols = k0 + nb
            add("potrf_diag_kernel", 2.0 * (nb ** 3 / 3 + nb ** 3 / 6))
            total = (2.0 * m * nb * nb + 2.0 * (m * (m + 1) / 2) * nb
                     + 2.0 * nb * ncols * nb + 2.0 * m * ncols * nb)
            chain = 0.0
            if m > 0:
                nn = min(NB, m)
                sp0 = k0 // spw * spw
                sp_end = min(d, sp0 + spw)
                ks = (sp_end - sp0) if k0 + nb == sp_end else nb
                chain = 2.0 * m * nb * nb + 2.0 * ks * (m * nn - nn * (nn - 1) / 2)
            add("tc_gemm_nt_kernel[chain]", chain)
            add("tc_gemm_nt_kernel[prepare]", total - chain)
            add("split_kernel", 12.0 * (m * nb + nb * ncols))
        for W in (L.Wcat,):   # one gptq_quantize per layer over the stacked weights
            r, c = W.shape
            add("split_kernel", 12.0 * c * c)
            add("init_work_kernel", 8.0 * r * c)
            for j0 in range(0, c, QB):
                bw = min(QB, c - j0)
                add("gptq_block_kernel", 2.0 * r * bw * bw)
                add("tc_gemm_nt_kernel[trailing]", 2.0 * r * bw * (c - j0 - bw))
            add("pack_kernel", r * c * 1.0 + r * -(-c * L.spec.q.bits // 32) * 4.0)
    return work


# kernel class -> (bound, unit); "tensor-tf32x3" is the fp32-accurate 3xTF32 product whose
# ceiling is the TF32 tensor peak / 3 (the TF32 peak measured in this run with a cuBLAS TF32
# GEMM, else GB300's nominal dense TF32:BF16 ratio of 1.1 : 2.25 times the measured bf16
# peak); "alu" kernels are measured against the FP32 FFMA peak
ROOF = {
    "hessian_tc_kernel": ("tensor", "TFLOP/s"),
    "tc_gemm_nt_kernel[prepare]": ("tensor-tf32x3", "TFLOP/s"),
    "tc_gemm_nt_kernel[chain]": ("tensor-tf32x3", "TFLOP/s"),
    "tc_gemm_nt_kernel[trailing]": ("tensor-tf32x3", "TFLOP/s"),
    "sgemm_kernel[prepare]": ("alu", "TFLOP/s"),
    "sgemm_kernel[trailing]": ("alu", "TFLOP/s"),
    "potrf_diag_kernel": ("alu", "TFLOP/s"),
    "gptq_block_kernel": ("alu", "TFLOP/s"),
    "pack_kernel": ("hbm", "GB/s"),
    "split_kernel": ("hbm", "GB/s"),
    "init_work_kernel": ("hbm", "GB/s"),
}

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the current kernels
# from the ncu captures of the Hessian kernel summarised under profiles/ (d = 4096 on 262144
# tokens, d = 14336 on 16384 tokens); a kernel changed since its capture has no entry here.
# The d = 14336 launch of the decoder block is estimated from its 16384-token capture: its
# reads (X re-streamed by each wave of tiles) scale with the tokens (x16), its writes (the
# accumulator flushes into S, one per tile) do not. Per launch, as `achieved` is.
_H4096 = 4.635595e9 + 160.0128e6
_H14336 = 4.726530e9 * 16 + 409.165056e6
TRAFFIC = {
    (2, "hessian_tc_kernel"): _H4096,
    (3, "hessian_tc_kernel"): _H14336,
    (4, "hessian_tc_kernel"): (3 * _H4096 + _H14336) / 4,
}


def peak_for(bound, pk, sustained: bool = False):
    """The roofline denominator of a kernel class. Tensor peaks are the burst figures for a
    short timed region and the sustained ones (seconds of back-to-back GEMMs under the power
    cap) for a timed region of a second or more; the TF32 sustained figure is the measured
    TF32 burst scaled by the measured bf16 sustained/burst ratio."""
    ratio = (pk["bf16_tflops_sustained"] / pk["bf16_tflops"]) if (sustained and pk.get("bf16_tflops_sustained")) else 1.0
    kind = "sustained" if ratio != 1.0 else "burst"
    if bound == "tensor":
        return pk["bf16_tflops"] * ratio, f"measured bf16 dense (cuBLAS {kind})"
    if bound == "tensor-tf32x3":
        if pk.get("tf32_tflops"):
            return (pk["tf32_tflops"] * ratio / 3.0,
                    f"measured TF32 dense (cuBLAS TF32 8192^3, this run; {kind}) / 3 passes")
        return (pk["bf16_tflops"] * ratio * (1.1 / 2.25) / 3.0,
                f"measured bf16 {kind} x 1.1/2.25 (GB300 nominal dense TF32:BF16) / 3")
    if bound == "alu":
        return FFMA_PEAK_TFLOPS, "derived: 152 SMs x 128 FP32 lanes x 2 x 2.07 GHz"
    return pk["hbm_gbs"], "measured HBM copy"


def measure_tf32_peak(dev, n: int = 8192, reps: int = 10) -> float:
    """Dense TF32 tensor-core throughput of a cuBLAS GEMM (fp32 in and out, TF32 products)
    on this GPU: the best of `reps` CUDA-event-timed n^3 products, in TFLOP/s."""
    import torch
    prev = torch.get_float32_matmul_precision()
    torch.set_float32_matmul_precision("high")   # fp32 matmuls on the TF32 tensor path
    try:
        a = torch.randn(n, n, device=dev)
        b = torch.randn(n, n, device=dev)
        c = torch.empty(n, n, device=dev)
        for _ in range(3):
            torch.matmul(a, b, out=c)
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b, c
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    finally:
        torch.set_float32_matmul_precision(prev)


# ------------------------------------------------------------------------- CPU oracle
#
# The oracle (numpy fp64, test infrastructure) timed on this host's cores, for context:
#   cpu_baseline (our arm, rank 0, N = 1): "one stated layer" timed whole - the whole
#     layer pass for the tiny and OPT workloads, the one layer of the Llama-7B attention
#     workload, and q_proj at 4 bits (H from the q/k/v input) for the decoder block; the
#     MLP-down layer (d = 14336) is too large for a whole CPU pass and is sampled (stated).
#     The column loop's rows are split over spawned processes (rows are independent given
#     U); H and U use the threaded BLAS/LAPACK of numpy.
#   reference arm: per step a bounded sample of the same stated layer (H on one 2048-token
#     segment, U in full, the loop on a few rows), timed as it runs - no scaling.

def stated_layer(cfg: int, wl):
    """(layer index, weight index) of the layer the CPU oracle times, or None for the whole
    layer pass (tiny and OPT workloads)."""
    if cfg in (0, 1):
        return None
    if cfg == 4:
        for li, L in enumerate(wl.layers):
            if L.q.bits == 4 and L.weights[0].name == "q_proj":
                return li, 0
    return 0, 0


def stated_desc(cfg: int, wl) -> str:
    st = stated_layer(cfg, wl)
    if st is None:
        return f"the whole {wl.name} layer pass"
    L = wl.layers[st[0]]
    w = L.weights[st[1]]
    return (f"{w.name} {w.out}x{w.inp} at {L.q.bits} bits (group {L.q.group}, "
            f"{'sym' if L.q.sym else 'asym'}{', act_order' if L.q.act_order else ''}) with H from its "
            f"{L.x.n}x{L.x.d} input")


# the reference arm's per-step sample: (tokens for H, rows of the column loop); U in full
REF_SAMPLE = {2: (2048, 8), 3: (2048, 4), 4: (2048, 8)}
# the MLP-down layer's CPU baseline: token and row fractions (timed parts scaled up)
CPU_SAMPLED = {3: (1.0 / 64, 1.0 / 256)}


def _oracle_rows_job(job):
    """Spawned worker: the oracle's quantisation of rows [r0, r1) of one weight given
    (U, perm, dead) saved under `folder` (rows are independent given U). Returns seconds."""
    folder, r0, r1, bits, group, sym = job
    import numpy as np
    import oracle as O
    if r1 <= r0:
        return 0.0
    U = np.load(os.path.join(folder, "U.npy"), mmap_mode="r")
    W = np.load(os.path.join(folder, "W.npy"), mmap_mode="r")
    perm = np.load(os.path.join(folder, "perm.npy"))
    dead = np.load(os.path.join(folder, "dead.npy"))
    t0 = time.perf_counter()
    O.gptq_quantize(np.array(W[r0:r1]), U, perm, dead, bits, group, sym)
    return time.perf_counter() - t0


def _noop_job(_):
    import numpy  # noqa: F401
    import oracle  # noqa: F401
    return 0


class RowPool:
    """A pool of spawned single-threaded processes for the oracle's column loop (spawn, not
    fork: the parent holds a CUDA context)."""

    def __init__(self, procs: int):
        import multiprocessing as mp
        keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
        old = {k: os.environ.get(k) for k in keys}
        for k in keys:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(procs)
            self.pool.map(_noop_job, range(procs))   # start-up and imports, untimed
        finally:
            for k, v in old.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.procs = procs

    def quantize(self, W, U, perm, dead, q) -> float:
        """Wall seconds of the oracle's gptq_quantize over all rows of W, split by rows."""
        import numpy as np
        folder = tempfile.mkdtemp(prefix="oracle_rows_")
        try:
            t0 = time.perf_counter()
            np.save(os.path.join(folder, "U.npy"), np.asarray(U, dtype=np.float64))
            np.save(os.path.join(folder, "W.npy"), np.asarray(W, dtype=np.float64))
            np.save(os.path.join(folder, "perm.npy"), np.asarray(perm))
            np.save(os.path.join(folder, "dead.npy"), np.asarray(dead))
            rows = W.shape[0]
            cuts = [rows * i // self.procs for i in range(self.procs + 1)]
            jobs = [(folder, cuts[i], cuts[i + 1], q.bits, q.group, q.sym) for i in range(self.procs)]
            self.pool.map(_oracle_rows_job, jobs)
            return time.perf_counter() - t0
        finally:
            for f in os.listdir(folder):
                os.unlink(os.path.join(folder, f))
            os.rmdir(folder)

    def close(self):
        self.pool.close()
        self.pool.join()


def oracle_pass(cfg: int, layers_host):
    """One layer pass of the oracle (numpy fp64) over host copies of the inputs; returns
    (ms for H over the tokens given, ms for the dead fix + damping + inv + cholesky, ms for
    the column loops + packing on the rows given)."""
    import numpy as np
    import oracle as O
    t_h = t_p = t_q = 0.0
    cache = {}
    for X, n_full, Ws, q in layers_host:
        key = (id(X), q.damp, q.act_order)   # shared inputs: H and U once, as on the GPU
        t0 = time.perf_counter()
        if key not in cache:
            S = O.xtx(X) * (n_full / X.shape[0])  # the sum over the sample, scaled to n tokens
            H = O.hessian_from_sum(S, n_full)
            t1 = time.perf_counter()
            cache[key] = O.prepare(H, q.damp, q.act_order, np.diag(S))
        else:
            t1 = t0
        U, perm, dead = cache[key]
        t2 = time.perf_counter()
        for W in Ws:
            O.gptq_quantize(W, U, perm, dead, q.bits, q.group, q.sym)
        t3 = time.perf_counter()
        t_h += (t1 - t0) * 1e3
        t_p += (t2 - t1) * 1e3
        t_q += (t3 - t2) * 1e3
    return t_h, t_p, t_q


def host_layers(layers):
    """Host fp64 copies of every layer's input and weights (one copy per distinct input)."""
    import synth
    out, xs = [], {}
    for L in layers:
        if id(L.X) not in xs:
            xs[id(L.X)] = synth.to_numpy_f64(L.X)
        out.append((xs[id(L.X)], L.X.shape[0], [synth.to_numpy_f64(W) for W in L.Ws], L.spec.q))
    return out


def oracle_stated_layer(cfg: int, wl, X, W, q, pool: "RowPool", token_frac: float = 1.0, row_frac: float = 1.0):
    """The oracle on one stated layer: S = sum over 2048-token segments of X_b^T X_b (each
    segment copied from X, a device or host tensor, to host fp64), H = 2 S / n, U, perm, dead,
    then the column loop over W's rows in the process pool. With token/row fractions below 1
    only that share is run and its time scaled up (stated in the description).
    Returns (total ms, {stage: ms})."""
    import numpy as np
    import oracle as O
    import synth
    n, d = X.shape
    seg = 2048
    n_s = max(1, int(round(n * token_frac)))
    t0 = time.perf_counter()
    S = None
    for r in range(0, n_s, seg):
        Xb = synth.to_numpy_f64(X[r:min(n_s, r + seg)])
        S = O.xtx(Xb) if S is None else S + O.xtx(Xb)
    S = S * (n / n_s)
    H = O.hessian_from_sum(S, n)
    t1 = time.perf_counter()
    U, perm, dead = O.prepare(H, q.damp, q.act_order, np.diag(S))
    t2 = time.perf_counter()
    rows = W.shape[0]
    r_s = max(pool.procs, int(round(rows * row_frac)))
    Wh = synth.to_numpy_f64(W[:r_s])
    tq = pool.quantize(Wh, U, perm, dead, q)
    # the same loop in this one process on a few rows (the P = 1 figure: ms per row)
    k = min(8, r_s)
    t3 = time.perf_counter()
    O.gptq_quantize(Wh[:k], U, perm, dead, q.bits, q.group, q.sym)
    p1_row = (time.perf_counter() - t3) / k
    th, tp = (t1 - t0) / (n_s / n), t2 - t1
    pool_row = tq / r_s
    tq = tq * rows / r_s
    comp = {"hessian": th * 1e3, "prepare": tp * 1e3, "quantize": tq * 1e3,
            "quantize_ms_per_row": {"processes": pool.procs, "pooled": pool_row * 1e3, "one_process": p1_row * 1e3,
                                    "one_process_rows_timed": k}}
    return (th + tp + tq) * 1e3, comp


def reference_sample(cfg: int, wl, device="cpu"):
    """Host inputs of the reference arm's per-step sample (generated on `device` from the
    workload's seeds; on the CPU the generator differs from the GPU's but the shapes and
    distributions are the same): the whole pass for the tiny and OPT workloads, else the
    stated layer's first 2048-token segment and its first few weight rows."""
    import synth
    if cfg in (0, 1):
        _, layers = build_layers(cfg, device)
        return {"kind": "whole", "layers": host_layers(layers),
                "desc": f"the whole {wl.name} layer pass in the oracle (numpy fp64), timed per step"}
    li, wi = stated_layer(cfg, wl)
    L = wl.layers[li]
    w = L.weights[wi]
    n_s, r_s = REF_SAMPLE[cfg]
    X = synth.make_x_rows(L.x, synth.x_seed(cfg, L.x), 0, n_s, device)
    W = synth.make_weight(w.out, w.inp, w.std, synth.weight_seed(cfg, w.name), device=device)[:r_s]
    return {"kind": "stated", "X": synth.to_numpy_f64(X), "n": L.x.n, "W": synth.to_numpy_f64(W), "q": L.q,
            "rows": w.out,
            "desc": (f"{stated_desc(cfg, wl)}: H on its first {n_s} tokens (S scaled to n = {L.x.n}), U in full, "
                     f"the column loop and packing on its first {r_s} of {w.out} rows; timed per step as run, "
                     "no scaling (one process, threaded BLAS)")}


def reference_step(sample):
    """One step of the reference arm's sample; returns (ms, {stage: ms})."""
    if sample["kind"] == "whole":
        t_h, t_p, t_q = oracle_pass(0, sample["layers"])
        return t_h + t_p + t_q, {"hessian": t_h, "prepare": t_p, "quantize": t_q}
    t_h, t_p, t_q = oracle_pass(0, [(sample["X"], sample["n"], [sample["W"]], sample["q"])])
    return t_h + t_p + t_q, {"hessian": t_h, "prepare": t_p, "quantize": t_q}


def bench_config(cfg: int, wl, ws: int) -> dict:
    """The `config` object of both arms' JSON lines (a function of the workload alone)."""
    xs = {}
    wbytes = 0
    for li, L in enumerate(wl.layers):
        xs[(L.x, x_group(cfg, wl, li))] = L.x.n * L.x.d * (2 if L.x.dtype == "bf16" else 4)
        wbytes += sum(w.out * w.inp * 4 for w in L.weights)
    in_bytes = sum(xs.values()) + wbytes
    flush = in_bytes < 2 * L2_BYTES
    return {"workload": wl.name, "config_index": cfg,
            "layers": [[[w.name for w in L.weights], [L.x.n, L.x.d], L.q.bits] for L in wl.layers],
            "input_bytes": in_bytes,
            "l2": ("flushed between steps (512 MiB write)" if flush else "inputs larger than L2"),
            "parallelism": f"replicas x{ws}", "stated_layer": stated_desc(cfg, wl)}


# ------------------------------------------------------------------------------ arms

def run_reference(args, ws, rank):
    if rank != 0:
        return
    import synth
    cores = len(os.sched_getaffinity(0))
    wl = workload_for(args)
    sample = reference_sample(args.config, wl)
    for _ in range(args.warmup):
        reference_step(sample)
    ts, comps = [], []
    t_wall = time.perf_counter()
    for _ in range(args.steps):
        t, c = reference_step(sample)
        ts.append(t)
        comps.append(c)
    wall = (time.perf_counter() - t_wall) * 1e3
    v = statistics.mean(ts)
    comp = {k: statistics.mean(c[k] for c in comps) for k in comps[0]}
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "ms", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": v, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": bench_config(args.config, wl, ws),
        "sample": sample["desc"], "components_ms": comp, "wall_ms_timed_region": wall,
        "cpu_baseline": {"value": v, "unit": "ms", "cores": cores, "kind": "oracle", "sample": sample["desc"]},
        "e2e": {"value": v, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    if sample["kind"] == "stated":
        n_s = sample["X"].shape[0]
        r_s = sample["W"].shape[0]
        line["extrapolated_stated_layer_ms"] = (comp["hessian"] * sample["n"] / n_s + comp["prepare"]
                                                + comp["quantize"] * sample["rows"] / r_s)
        line["extrapolation"] = ("not measured: the sample's H time x n/tokens + prepare + loop time x "
                                 "rows/sampled rows, one process")
    print(json.dumps(line), flush=True)


def max_over_ranks(ms: float, ws: int, device) -> float:
    """The slowest rank's step time (every rank gets it)."""
    if ws <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(ms_max: float, ws: int) -> float:
    """ws independent replicas each finish one layer pass within ms_max: the job's time per
    layer pass (weak scaling; lower is better)."""
    return ms_max / max(1, ws)


def run_ours(args, ws, rank, local):
    import torch
    import torch.distributed as dist
    import post_weight_quantization_04_gb300 as lib
    from post_weight_quantization_04_gb300 import build as B

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    B.build()
    lib.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pk = peaks()
    pk["tf32_tflops"] = measure_tf32_peak(dev)
    pk["tf32_source"] = "cuBLAS TF32 GEMM 8192^3, best of 10, CUDA events, this run"

    wl, layers = build_layers(args.config, dev, wl=workload_for(args))
    runner = Runner(lib, layers, dev)
    # deferred status reporting: the calls of a step only enqueue work (no host round trip
    # between them); device-side errors are checked once per step with status_sync
    lib.set_status_mode(True)
    flush = bench_config(args.config, wl, ws)["input_bytes"] < 2 * L2_BYTES
    fbuf = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev) if flush else None

    def barrier():
        if ws > 1:
            dist.barrier()

    # clocks are sampled every 200 ms from before the warm-up to the end of the timed
    # region (at the small workloads the timed region itself is a few milliseconds)
    def run_step():
        if args.schedule == "serial":
            return runner.step()
        return runner.step_concurrent(quantize_in_group=(args.schedule in ("groups", "layers")),
                                      fork_layers=(args.schedule == "layers"))

    clocks = Clocks(local)
    clocks.start()
    for _ in range(args.warmup):
        run_step()
    lib.status_sync()
    torch.cuda.synchronize()

    # The step's library calls captured once into a CUDA graph (in the deferred status mode
    # they only enqueue work) and replayed: every replay runs every kernel of the step on
    # the same resident inputs, without the host launch overhead between them.
    graph, graph_launches, graph_note = None, 0, None
    if not args.no_graph:
        try:
            gs = torch.cuda.Stream()
            gs.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(gs):
                run_step()
                lib.status_sync(gs)
            torch.cuda.current_stream().wait_stream(gs)
            graph = torch.cuda.CUDAGraph()
            c0 = lib.gptq_launch_count()
            with torch.cuda.graph(graph, stream=gs):
                run_step()
            graph_launches = lib.gptq_launch_count() - c0
            graph.replay()
            lib.status_sync()
            torch.cuda.synchronize()
        except Exception as e:  # noqa: BLE001  (a capture the runtime refuses: time eager calls)
            graph, graph_note = None, f"graph capture failed ({type(e).__name__}); eager calls"
            torch.cuda.synchronize()
            lib.status_sync()

    barrier()
    torch.cuda.synchronize()
    n0 = lib.gptq_launch_count()
    times = []
    t_wall0 = time.perf_counter()
    for _ in range(args.steps):
        if flush:
            flush_l2(fbuf)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        if graph is not None:
            graph.replay()
        else:
            run_step()
        b.record()
        lib.status_sync()   # synchronises the stream: the step's errors, after its end event
        times.append(a.elapsed_time(b))
    torch.cuda.synchronize()
    barrier()
    wall = (time.perf_counter() - t_wall0) * 1e3
    # a replay launches the graph's kernels without passing the library's launch counter
    launches = graph_launches * args.steps if graph is not None else lib.gptq_launch_count() - n0
    ck = clocks.stop()
    ms = max_over_ranks(statistics.mean(times), ws, dev)

    # ---- profiled pass: per-stage and per-kernel CUDA events over the same steps ----
    # a timed region of a second or more keeps the tensor cores loaded long enough for the
    # power cap to act: its kernels are measured against the sustained tensor peaks
    long_region = sum(times) >= 1000.0
    stages, kernels, roof = {}, {}, None
    if not args.no_profile:
        # stage times from serial steps with events only between the calls (the library's
        # per-launch profiling below would break programmatic dependent launch inside them)
        evs = []
        for _ in range(args.steps):
            if flush:
                flush_l2(fbuf)
            runner.step(events=evs)
            lib.status_sync()
        torch.cuda.synchronize()
        for name, idx in (("hessian", (0, 1)), ("prepare", (1, 2)), ("quantize", (2, 3))):
            stages[name] = sum(e[idx[0]].elapsed_time(e[idx[1]]) for e in evs) / args.steps
        stages["serial_step"] = sum(e[0].elapsed_time(e[3]) for e in evs) / args.steps
        stages["per_group"], stages["per_bits"] = stage_breakdown(evs, runner.groups, layers, args.steps)
        lib.gptq_profile_enable(True)
        lib.gptq_profile_read()
        for _ in range(args.steps):
            if flush:
                flush_l2(fbuf)
            runner.step()
            lib.status_sync()
        torch.cuda.synchronize()
        lib.gptq_profile_enable(False)
        prof = lib.gptq_profile_read()
        tot = sum(v[1] for v in prof.values())
        work = algorithmic(layers)
        for name, (cnt, t) in sorted(prof.items(), key=lambda kv: -kv[1][1]):
            kernels[name] = {"launches_per_step": cnt / args.steps, "ms_per_step": t / args.steps,
                             "share": t / tot if tot else None}
            if name in work and name in ROOF:
                bound, unit = ROOF[name]
                sec = t / args.steps / 1e3
                peak, src = peak_for(bound, pk, sustained=long_region)
                ach = work[name] / sec / (1e12 if unit == "TFLOP/s" else 1e9)
                kernels[name].update({"bound": bound, "achieved": ach, "peak": peak, "unit": unit,
                                      "frac": ach / peak, "peak_source": src})
            if name == "gptq_block_kernel":
                # the loop's sequential chain: time per column of the stacked weights (each
                # call walks its columns once, all rows in parallel)
                ncols = sum(L.Wcat.shape[1] for L in layers)
                kernels[name]["ns_per_column"] = t / args.steps * 1e6 / ncols
        top = max(kernels.items(), key=lambda kv: kv[1]["ms_per_step"])[0] if kernels else None
        if top:
            k = kernels[top]
            per_launch = k["ms_per_step"] / max(1.0, k["launches_per_step"])
            roof = {"kernel": top, "bound": k.get("bound"), "achieved": k.get("achieved"), "peak": k.get("peak"),
                    "unit": k.get("unit"), "frac": k.get("frac"),
                    "traffic": TRAFFIC.get((args.config, top)), "peak_source": k.get("peak_source"),
                    "avg_launch_ms": per_launch}
        if "hessian_tc_kernel" in kernels:
            stages["hessian_tc_frac_of_bf16_peak"] = kernels["hessian_tc_kernel"].get("frac")
            k = kernels["hessian_tc_kernel"]
            stages["hessian_tc_frac_of_bf16_burst_peak"] = k.get("achieved", 0.0) / pk["bf16_tflops"]

    # ---- e2e: pinned host inputs -> device -> same pass -> quantised artefacts back ----
    e2e = None
    if not args.no_e2e:
        # one host copy and one device buffer per distinct X (shared inputs are copied once)
        xs = {}
        for L in layers:
            if id(L.X) not in xs:
                hx = torch.empty(L.X.shape, dtype=L.X.dtype, pin_memory=True)
                hx.copy_(L.X)
                xs[id(L.X)] = (hx, torch.empty_like(L.X))
        hX = [v[0] for v in xs.values()]
        dXu = [v[1] for v in xs.values()]
        dX = [xs[id(L.X)][1] for L in layers]
        hW = [torch.empty(L.Wcat.shape, dtype=L.Wcat.dtype, pin_memory=True).copy_(L.Wcat) for L in layers]
        dW = [torch.empty_like(L.Wcat) for L in layers]
        h_out = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in o.items()
                  if k in ("packed", "scales", "zeros", "g_idx")} for o in runner.outs]
        bi = sum(x.numel() * x.element_size() for x in hX) + sum(w.numel() * 4 for w in hW)
        bo = sum(v.numel() * v.element_size() for o in h_out for v in o.values())

        # The copies run on their own streams, overlapped with the pass (host-to-device
        # bandwidth, not the pass, would otherwise set the step). The groups run largest
        # input first; each input is copied in token chunks on a copy stream and
        # its Hessian accumulates each chunk as soon as it has landed, so the largest copy
        # hides behind the largest Hessian and the smaller groups' copies land while the
        # first group is factorised and quantised. Each layer's weights are copied right
        # after its group's input (the pass waits for them just before the layer), and each
        # layer's stored form goes back on a second stream as soon as the layer is done.
        # Inputs are cut into one chunk per 256 MB, at most 8 (a small input stays whole:
        # its extra Hessian launches would cost more than the copy they overlap).
        h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
        link = settle_host_link(torch, h2d, [(dx, hx) for hx, dx in xs.values()] + list(zip(dW, hW)))
        gorder = sorted(range(len(runner.groups)),
                        key=lambda gi: -layers[runner.groups[gi][0]].X.numel() * layers[runner.groups[gi][0]].X.element_size())
        x_chunks = {}
        for gi, g in enumerate(runner.groups):
            dx = dX[g[0]]
            n = dx.shape[0]
            nch = max(1, min(8, (dx.numel() * dx.element_size()) // (256 << 20)))
            cuts = [n * c // nch for c in range(nch + 1)]
            x_chunks[gi] = [(dx[cuts[c]:cuts[c + 1]], torch.cuda.Event(), cuts[c]) for c in range(nch)
                            if cuts[c + 1] > cuts[c]]
        w_ready = [torch.cuda.Event() for _ in layers]
        layer_done = [torch.cuda.Event() for _ in layers]

        def e2e_enqueue():
            main = torch.cuda.current_stream()
            h2d.wait_stream(main)
            d2h.wait_stream(main)
            copied = {}
            with torch.cuda.stream(h2d):
                for gi in gorder:
                    g = runner.groups[gi]
                    key = id(layers[g[0]].X)
                    hx, dx = xs[key]
                    if key not in copied:
                        copied[key] = gi
                        for rows, ev, r0 in x_chunks[gi]:
                            rows.copy_(hx[r0:r0 + rows.shape[0]], non_blocking=True)
                            ev.record()
                    else:   # an input shared with an earlier group: its chunks are in already
                        for rows, ev, r0 in x_chunks[gi]:
                            ev.record()
                    for li in g:
                        dW[li].copy_(hW[li], non_blocking=True)
                        w_ready[li].record()
            kw = dict(Xs=dX, Wcats=dW, x_chunks=x_chunks, w_ready=w_ready, layer_done=layer_done, order=gorder)
            outs = (runner.step(**kw) if args.schedule == "serial"
                    else runner.step_concurrent(quantize_in_group=(args.schedule in ("groups", "layers")),
                                                fork_layers=(args.schedule == "layers"), **kw))
            with torch.cuda.stream(d2h):
                for gi in gorder:
                    for li in runner.groups[gi]:
                        d2h.wait_event(layer_done[li])
                        for k in h_out[li]:
                            h_out[li][k].copy_(outs[li][k], non_blocking=True)
            main.wait_stream(d2h)

        def e2e_step():
            e2e_enqueue()
            lib.status_sync()   # synchronises the stream, then raises on a device-side error

        for _ in range(max(1, args.warmup)):
            e2e_step()
        # the same calls and copies captured once into a CUDA graph (as the device-timed step
        # is): a replay enqueues the step's ~2800 launches and its copies at once, so the
        # host's own speed at issuing them drops out of the timed region
        egraph, e_note = None, None
        if not args.no_graph:
            try:
                cs = torch.cuda.Stream()
                cs.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(cs):
                    e2e_enqueue()
                    lib.status_sync(cs)
                torch.cuda.current_stream().wait_stream(cs)
                egraph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(egraph, stream=cs):
                    e2e_enqueue()
                egraph.replay()
                lib.status_sync()
                torch.cuda.synchronize()
            except Exception as e:  # noqa: BLE001  (a capture the runtime refuses: time eager calls)
                egraph, e_note = None, f"graph capture failed ({type(e).__name__}); eager calls"
                torch.cuda.synchronize()
                lib.status_sync()
        et = []
        for _ in range(args.steps):
            if flush:
                flush_l2(fbuf)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            if egraph is not None:
                egraph.replay()
                lib.status_sync()
            else:
                e2e_step()
            et.append((time.perf_counter() - t0) * 1e3)
        # the same step issued call by call from the host (for comparison)
        eager = []
        for _ in range(3):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            e2e_step()
            eager.append((time.perf_counter() - t0) * 1e3)
        # the step's host-to-device copies alone (the floor the host link sets on e2e)
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(h2d):
            c0.record()
            for hx, dx in xs.values():
                dx.copy_(hx, non_blocking=True)
            for li in range(len(layers)):
                dW[li].copy_(hW[li], non_blocking=True)
            c1.record()
        torch.cuda.synchronize()
        e2e = {"value": statistics.mean(et), "unit": "ms", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
               "h2d_alone_ms": c0.elapsed_time(c1), "host_link": link,
               "step": ("one CUDA graph of the copies and library calls, replayed" if egraph is not None
                        else e_note or "the copies and library calls issued eagerly"),
               "eager_ms": statistics.mean(eager),
               "copies": "pinned host buffers; the inputs go in on a copy stream in token chunks (one per 256 MB, at "
                         "most 8), largest input first, each chunk accumulated into its Hessian once landed; weights "
                         "follow their group's input; each layer's stored form goes back on another stream once the "
                         "layer is done"}

    # ---- the stated layer on the GPU (the layer the CPU oracle times whole) ----
    stated = stated_layer(args.config, wl)
    gpu_stated_ms = ms if stated is None else time_stated_layer_gpu(lib, runner, layers, stated, dev)

    # ---- CPU oracle baseline (rank 0, N = 1 only) ----
    cpu = None
    if not args.no_cpu_baseline and rank == 0 and ws == 1:
        cpu = cpu_baseline(args.config, wl, layers)

    if rank == 0:
        value = replica_value(ms, ws)
        line = {
            "metric": METRIC, "value": value, "unit": "ms", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "s_per_step": ms / 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16xbf16->f32 (Hessian), f32 (rest)",
            "data": "synthetic", "config": bench_config(args.config, wl, ws),
            "step": ("one CUDA graph of the step's library calls, replayed" if graph is not None
                     else graph_note or "the library calls issued eagerly"),
            "schedule": {"serial": "group after group",
                         "prepare": "all Hessians, then every group's gptq_prepare side by side on its own stream, "
                                    "then the quantizations",
                         "groups": "all Hessians, then per group on its own stream its gptq_prepare and its "
                                   "gptq_quantize calls, the groups side by side",
                         "layers": "all Hessians, then per group on its own stream its gptq_prepare, then each "
                                   "of its layers' gptq_quantize on a stream of its own, all side by side"
                         }[args.schedule],
            "clocks": ck, "gpu_launches": launches // max(1, args.steps) * args.steps,
            "gpu_launches_per_step": launches / max(1, args.steps), "wall_ms_timed_region": wall,
            "stages_ms": stages, "kernels": kernels, "roofline": roof, "e2e": e2e, "cpu_baseline": cpu,
            "stated_layer": {"what": stated_desc(args.config, wl), "gpu_ms": gpu_stated_ms,
                             "cpu_ms": cpu["value"] if cpu else None},
            "peaks": pk,
        }
        print(json.dumps(line), flush=True)


def time_stated_layer_gpu(lib, runner, layers, stated, dev, reps: int = 5) -> float:
    """Device time (CUDA events, mean of `reps` after one warm-up) of the stated layer alone:
    one Hessian pass over its input, gptq_prepare, and gptq_quantize of that one weight."""
    import torch
    li, wi = stated
    L = layers[li]
    W = L.Ws[wi]
    grp = next(g for g in runner.groups if li in g)
    q = L.spec.q
    h = runner.hess[L.X.shape[1]]
    ws_q = torch.empty(lib.gptq_quantize_workspace_bytes(W.shape[0], W.shape[1], q.bits, q.group, q.sym),
                       dtype=torch.uint8, device=dev)

    def one():
        h.reset()
        h.accumulate(L.X)
        H, diag, _ = h.finalize()
        U, perm, dead = lib.gptq_prepare(H, diag, q.damp, act_order=q.act_order, ws=runner.prep_ws[id(grp)])
        lib.gptq_quantize(W, U, perm, dead, q.bits, q.group, q.sym, ws=ws_q)

    one()
    lib.status_sync()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        one()
        b.record()
        lib.status_sync()
        ts.append(a.elapsed_time(b))
    return statistics.mean(ts)


def settle_host_link(torch, stream, copies, limit_s: float = 150.0) -> dict:
    """Wait (at most limit_s) until the host link copies at a steady rate: the step's own
    host-to-device copies (`copies`: (device, pinned host) pairs), timed pass after pass
    until two passes in a row take at most 25% longer than the fastest seen. Right after a
    process that used and freed tens of GB of host memory, the box's kernel migrates pages
    for minutes and copies drop to a fraction of the link's rate, some buffers at a time;
    the e2e timing waits that out instead of measuring it. Returns the passes' times and
    the wait."""
    t0 = time.perf_counter()
    passes = []
    steady = False
    while True:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record()
            for dst, src in copies:
                dst.copy_(src, non_blocking=True)
            b.record()
        b.synchronize()
        passes.append(a.elapsed_time(b))
        best = min(passes)
        steady = len(passes) >= 2 and max(passes[-2:]) <= 1.25 * best
        waited = time.perf_counter() - t0
        if steady or waited >= limit_s:
            break
    return {"passes": len(passes), "last_pass_ms": round(passes[-1], 1), "best_pass_ms": round(min(passes), 1),
            "steady": steady, "waited_s": round(waited, 1)}


def cpu_baseline(cfg: int, wl, layers) -> dict:
    """The oracle on this host's cores: the stated layer timed whole (sampled and scaled for
    the MLP-down layer, which says so), plus one step of the reference arm's sample."""
    cores = len(os.sched_getaffinity(0))
    st = stated_layer(cfg, wl)
    if st is None:
        t_h, t_p, t_q = oracle_pass(cfg, host_layers(layers))
        value, comp = t_h + t_p + t_q, {"hessian": t_h, "prepare": t_p, "quantize": t_q}
        desc = (f"the whole {wl.name} layer pass in the oracle (numpy fp64: H, inv + cholesky, column loop, "
                f"packing), one process with threaded BLAS/LAPACK on {cores} cores")
        used = cores
    else:
        li, wi = st
        L = layers[li]
        pool = RowPool(cores)
        try:
            tf, rf = CPU_SAMPLED.get(cfg, (1.0, 1.0))
            value, comp = oracle_stated_layer(cfg, wl, L.X, L.Ws[wi], L.spec.q, pool, tf, rf)
        finally:
            pool.close()
        used = cores
        if cfg in CPU_SAMPLED:
            desc = (f"{stated_desc(cfg, wl)} in the oracle (numpy fp64): H on the first {tf:.4g} of the tokens "
                    f"(time scaled by {1 / tf:.4g}), inv + cholesky in full, the column loop and packing on "
                    f"the first {rf:.4g} of the rows split over {cores} processes (time scaled by {1 / rf:.4g}); "
                    "a whole CPU pass of this layer takes tens of minutes")
        else:
            desc = (f"{stated_desc(cfg, wl)}, timed whole in the oracle (numpy fp64): H streamed over all "
                    f"{L.X.shape[0]} tokens in 2048-token segments and inv + cholesky with threaded "
                    f"BLAS/LAPACK on {cores} cores, the column loop and packing with the rows split over "
                    f"{cores} single-threaded processes (rows are independent given U)")
    out = {"value": value, "unit": "ms", "cores": used, "kind": "oracle", "sample": desc, "components_ms": comp}
    if st is not None:
        # one step of the reference arm's per-step sample, on the same host: the two arms'
        # CPU numbers for the same sample
        sample = reference_sample(cfg, wl)
        out["reference_sample_ms"], _ = reference_step(sample)
        out["reference_sample"] = sample["desc"]
    return out


def run_dequant_matmul(args):
    """Y = X Wq^T from the stored form of the workload's first stacked weight matrix (as
    gptq_quantize writes it), X = the first `tokens` rows of that layer's input. One JSON
    line: TFLOP/s against the measured bf16 peak, and the stored-weight bytes read."""
    import torch
    import post_weight_quantization_04_gb300 as lib
    from post_weight_quantization_04_gb300 import build as B

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    B.build()
    lib.load()
    dev = torch.device("cuda", 0)
    pk = peaks()
    wl, layers = build_layers(args.config, dev)
    L = layers[0]
    q = L.spec.q
    h = lib.Hessian(L.X.shape[1], dev)
    h.accumulate(L.X)
    H, diag, _ = h.finalize()
    U, perm, dead = lib.gptq_prepare(H, diag, q.damp, act_order=q.act_order)
    st = lib.gptq_quantize(L.Wcat, U, perm, dead, q.bits, q.group, q.sym)
    X = L.X[: args.tokens].contiguous()
    T, K = X.shape
    N = L.Wcat.shape[0]
    Y = torch.empty(T, N, dtype=torch.float32, device=dev)
    zeros = st["zeros"]

    def step():
        lib.gptq_dequant_matmul(X, st["packed"], st["scales"], zeros, st["g_idx"], q.bits, out=Y)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    n0 = lib.gptq_launch_count()
    times = []
    for _ in range(args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        step()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    ms = statistics.mean(times)
    flops = 2.0 * T * K * N
    tf = flops / (ms * 1e-3) / 1e12
    wbytes = st["packed"].numel() * 4 + st["scales"].numel() * 4 + zeros.numel()
    print(json.dumps({
        "metric": "dequant matmul from the stored form (TFLOP/s)", "value": tf, "unit": "TFLOP/s",
        "higher_is_better": True, "ms_per_step": ms, "steps": args.steps, "n_gpus": 1,
        "dtype": "bf16 x (b-bit -> bf16) -> f32", "data": "synthetic",
        "config": {"workload": wl.name, "tokens": T, "in": K, "out": N, "bits": q.bits, "group": q.group,
                   "act_order": q.act_order, "stored_weight_bytes": wbytes},
        "gpu_launches": lib.gptq_launch_count() - n0,
        "roofline": {"bound": "tensor", "achieved": tf, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": tf / pk["bf16_tflops"], "traffic": None},
    }), flush=True)


def run_quantize(args):
    """gptq_quantize alone on a rows x cols weight stack (--shape) with a synthetic,
    well-conditioned U (the loop's cost does not depend on U's values), bits --bits (else
    4), groups of 128, symmetric. One JSON line: ms per call (device time, CUDA events).
    The call's trailing updates are cols/128 - 1 launches of the 3xTF32 GEMM: per 512
    columns three inside the super-block (K = 128), then one over all columns past it
    (K = 512)."""
    import torch
    import post_weight_quantization_04_gb300 as lib
    from post_weight_quantization_04_gb300 import build as B

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    B.build()
    lib.load()
    dev = torch.device("cuda", 0)
    rows, cols = (int(v) for v in args.shape.lower().split("x"))
    bits = args.bits or 4
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    W = (torch.randn(rows, cols, device=dev, generator=g) * 0.02).contiguous()
    U = torch.triu(torch.randn(cols, cols, device=dev, generator=g) * (0.3 / cols ** 0.5), 1)
    U += torch.diag(torch.rand(cols, device=dev, generator=g) + 0.5)
    ws = torch.empty(lib.gptq_quantize_workspace_bytes(rows, cols, bits, 128, True), dtype=torch.uint8, device=dev)
    out = None

    def step():
        nonlocal out
        out = lib.gptq_quantize(W, U, None, None, bits, 128, True, ws=ws, out=out)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    n0 = lib.gptq_launch_count()
    times = []
    for _ in range(args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        step()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    print(json.dumps({
        "metric": "gptq_quantize (ms per call)", "value": statistics.mean(times), "unit": "ms",
        "higher_is_better": False, "steps": args.steps, "n_gpus": 1, "data": "synthetic",
        "dtype": "f32 (trailing updates 3xTF32)",
        "config": {"rows": rows, "cols": cols, "bits": bits, "group": 128, "sym": True},
        "gpu_launches": lib.gptq_launch_count() - n0,
    }), flush=True)


def run_layerwise(args):
    """The layer-wise pipeline on a synthetic MLP: per layer H from the previous quantised
    layers' bf16 outputs, prepare, quantize, and the forward pass on the stored form. One
    JSON line: ms per whole-network pass (device time, CUDA events)."""
    import torch
    import post_weight_quantization_04_gb300 as lib
    from post_weight_quantization_04_gb300 import build as B
    import synth

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    B.build()
    lib.load()
    dev = torch.device("cuda", 0)
    spec = synth.mlp_workload(args.mlp)
    X = synth.make_x(spec.x, 1234, device=dev)
    Ws = synth.make_mlp_weights(spec, 1334, device=dev)

    def step():
        return lib.gptq_layerwise(X, Ws, spec.bits, spec.group, spec.sym, spec.damp, spec.act_order)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    n0 = lib.gptq_launch_count()
    times = []
    for _ in range(args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        step()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    ms = statistics.mean(times)
    print(json.dumps({
        "metric": "layer-wise MLP quantization (ms per network pass)", "value": ms, "unit": "ms",
        "higher_is_better": False, "steps": args.steps, "n_gpus": 1, "data": "synthetic",
        "dtype": "bf16 activations, f32 quantisation", "config": {"workload": spec.name, "dims": list(spec.dims),
                                                                   "tokens": spec.x.n, "bits": spec.bits,
                                                                   "group": spec.group},
        "gpu_launches": (lib.gptq_launch_count() - n0) // max(1, args.steps) * args.steps,
    }), flush=True)


def main():
    # The concurrent step runs ~25 streams (groups, layers, the factorisation's own
    # streams). With the runtime's default of 8 hardware work queues, streams share queues
    # and unrelated work waits behind each other; 32 (the maximum) gives each its own. Read
    # when the CUDA context is created, so set before any CUDA call of this process.
    os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")
    args = parse()
    ws, rank, local = dist_info()
    if ws > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return
        else:
            dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.op == "dequant_matmul":
        if rank == 0:
            run_dequant_matmul(args)
    elif args.op == "layerwise":
        if rank == 0:
            run_layerwise(args)
    elif args.op == "quantize":
        if rank == 0:
            run_quantize(args)
    elif args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_ours(args, ws, rank, local)
    if ws > 1 and args.impl != "reference":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
