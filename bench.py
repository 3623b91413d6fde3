#!/usr/bin/env python
"""Benchmark of the virtual-noise ES step on one node.

Default workload (the headline): the large tensor-core forward, pop 256 x batch 256,
4096 -> 4096, X / W / Y bf16, sigma 0.01 -- one launch of the fused perturbed
linear (tcgen05 + TMEM) per step, 4.3e9 noise elements regenerated per step.
The same JSON line carries, under "configs", the other workloads measured the same
way with their own roofline objects:
  * mid:       pop 4096, batch 32, 1024 -> 1024 (X bf16, W fp32): the tensor-core
               forward plus grad_W and grad_b,
  * grad_only: grad_W and grad_b of a 4096 x 4096 block over pop 16384, fitness the
               centered ranks of the returns (the ranks computed on the device),
  * es_mlp:    one ES generation of the MLP policy (pop 1024, batch 1, 64 -> 256 ->
               256 -> 8 with tanh, fp32): the three layers in one launch, centered
               ranks, the flat gradient of all six blocks with the parameter step
               fused, and the noise dump of the whole parameter vector; its e2e is
               reported with and without the dump,
  * tiny:      pop 8, batch 4, 32 -> 16, fp32: forward, gradients and dump,
and "alu_peak_measured": the hash-only kernel (vn_hash_probe), whose element rate is
the measured ceiling of the integer ALU pipe beside the derived one.
`--workload NAME` makes another workload the headline (then no extras unless
`--extras` names them); `--noise gaussian` runs the Box-Muller variant of the noise
throughout.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl vn|reference]
                       [--workload large_tc|mid|grad_only|es_mlp|tiny] [--extras auto|none|a,b]
For N > 1 launch with torch.distributed.run: every rank runs its own population
(seeds offset by rank * pop), no data-path collective (weak scaling).

Timing: W untimed warm-up steps, then two timed passes between barriers and
device synchronisations, each rewriting a 256 MiB buffer between steps (outside
the events) so that every step starts with a cold L2:
  * the step pass: K steps, each bracketed by one pair of CUDA events on the
    launching stream -> ms_per_step and value. The step's C-ABI calls are
    captured once into a CUDA graph, replayed per step (--no-graph: direct calls);
  * the kernel pass: the same launches again (--kernel-steps, default K), every
    launch bracketed by its own pair of events -> per-kernel durations, shares
    and the dominant kernel's roofline. (An event pair around each launch adds
    its own gap between launches, so it is kept out of the step pass.)
The headline times exactly K steps; an extra workload times min(K, the steps that
fit --extra-seconds, at least 3) and says how many in its entry.
The oracle legs (cpu_baseline, --impl reference) run the oracle as it stands on
the host's cores: each individual's pass is independent, so the sampled
individuals are split over one spawned process per core.
Rank 0 prints one JSON line.
"""

from __future__ import annotations

import os

# The oracle legs report the threads they use: keep every BLAS / OpenMP pool at one.
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import ctypes
import hashlib
import json
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "virtual-noise elem/s"
UNIT = "noise elements/s"

# Cost of one noise element in the definition, on 32-bit halves (the GPU has no
# 64-bit integer unit). Integer ALU pipe (LOP3 / SHF / IADD3): right shifts 6 (two
# funnel shifts and two plain shifts for the xor-shifts 30 and 27, two for the
# final xor-shift 31 with the top-23-bit extraction), three-input logic ops 5, and
# the low word of the 64-bit state add 1 (its high word, an add with carry-in, can
# issue on the IMAD pipe, as the compiler does in the gradient kernel) -> 12. IMAD
# pipe: the two products by GAMMA, 3 each, plus that carry add -> 7. Plus the float
# conversion and the FMA that consumes the noise -> 21 operations in all.
ALU_OPS_PER_ELEMENT = 12
# The Gaussian variant: both halves of the last xor-shift and two mantissas
# (13 ALU operations in all, per ncu's per-opcode counts), three transcendental
# operations (log2, reciprocal square root, cos) and the floating-point glue of
# Box-Muller: about 32 instructions per element, so the issue port (4 schedulers
# x 32 lanes per SM) binds rather than the ALU pipe or the 32-lane MUFU pipe.
ALU_OPS_GAUSSIAN = 13
OPS_GAUSSIAN = 32
MUFU_OPS_GAUSSIAN = 3
MUFU_LANES_PER_SM = 32
OPS_PER_ELEMENT = 21
SMS_NOMINAL = 152
SM_CLOCK_MAX_HZ = 2.07e9
ALU_LANES_PER_SM = 64             # integer ALU pipe: 16 lanes per scheduler, 4 schedulers
ISSUE_LANES_PER_SM = 128          # 4 schedulers x 32 lanes, one instruction per clock each
L2_FLUSH_BYTES = 256 << 20
ES_LR = 0.01                      # learning rate of the bench's parameter update
E2E_SETS = 3                      # device buffer sets the e2e loop rotates through


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    p = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        p = {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
             "bf16_tflops_sustained": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])),
             "source": "measured"}
    p["alu_ops"] = SMS_NOMINAL * ALU_LANES_PER_SM * SM_CLOCK_MAX_HZ
    p["issue_ops"] = SMS_NOMINAL * ISSUE_LANES_PER_SM * SM_CLOCK_MAX_HZ
    return p


# ---------------------------------------------------------------------------
# Workload -> list of launches through the C ABI
# ---------------------------------------------------------------------------

class Launch:
    """One C-ABI call with its arguments fixed; ``kernel`` names the kernel it runs."""

    def __init__(self, kernel, fn, args, elements, flops=0.0, hbm_bytes=0.0, grad_w_elems=0):
        self.kernel, self.fn, self.args = kernel, fn, args
        self.elements, self.flops, self.hbm_bytes = elements, flops, hbm_bytes
        self.grad_w_elems = grad_w_elems

    def __call__(self):
        st = self.fn(*self.args)
        if st != 0:
            from virtual_noise_perturbed_gb300._lib import VNError
            raise VNError(st, self.kernel)


def contiguous_blocks(wl) -> bool:
    """True when the layers' blocks follow one another as compute_offsets lays them out."""
    off = wl.layers[0].offset
    for l in wl.layers:
        if l.offset != off:
            return False
        off += l.out_f * l.in_f + l.out_f
    return True


def build_step(wl, dev, stream_ptr, noise="uniform", include_dump=True):
    """Device buffers and the launches of one step of workload ``wl`` (on ``dev``);
    ``noise="gaussian"`` runs the step with the Box-Muller variant of the noise;
    ``include_dump=False`` leaves the noise dump of the tiny and policy workloads out."""
    import torch
    from virtual_noise_perturbed_gb300 import _lib

    lib = _lib.load()
    P = ctypes.c_void_p
    s = P(stream_ptr)
    d = wl.to(dev)
    bufs = {"seeds": d.seeds}
    launches = []
    outputs = []
    pop, batch = wl.pop, wl.batch
    dt = {torch.float32: _lib.VN_F32, torch.bfloat16: _lib.VN_BF16}
    n_params = sum(l.out_f * l.in_f + l.out_f for l in wl.layers)
    flat = wl.grads and len(wl.layers) > 1 and contiguous_blocks(wl)
    suffix = "_gaussian" if noise == "gaussian" else ""

    fused = (wl.forward and len(d.layers) > 1 and batch <= 8 and d.x.dtype in (torch.float32, torch.bfloat16)
             and all(l.weight.dtype == torch.float32 and l.bias.dtype == torch.float32 for l in d.layers))
    theta = None
    if fused and flat:
        # One flat parameter vector (W_0, b_0, W_1, b_1, ... as compute_offsets lays
        # them out); the layers are views of it, so the update is one launch.
        theta = torch.cat([t.reshape(-1) for l in d.layers for t in (l.weight, l.bias)]).contiguous()
        pos = 0
        for l in d.layers:
            l.weight = theta[pos:pos + l.out_f * l.in_f].view(l.out_f, l.in_f)
            pos += l.out_f * l.in_f
            l.bias = theta[pos:pos + l.out_f]
            pos += l.out_f
        bufs["theta"] = theta
    if fused:
        # A policy (several fp32 layers, small batch): every layer in one launch,
        # the activations kept on chip (vn_perturbed_mlp).
        bufs["x"] = d.x
        n = len(d.layers)
        dims = [d.layers[0].in_f] + [l.out_f for l in d.layers]
        if theta is None:
            for li, l in enumerate(d.layers):
                bufs[f"w{li}"], bufs[f"b{li}"] = l.weight, l.bias
        y = torch.empty((pop, batch, dims[-1]), dtype=torch.float32, device=dev)
        c_dims = (ctypes.c_int64 * (n + 1))(*dims)
        c_w = (ctypes.c_void_p * n)(*[l.weight.data_ptr() for l in d.layers])
        c_b = (ctypes.c_void_p * n)(*[l.bias.data_ptr() for l in d.layers])
        c_off = (ctypes.c_uint64 * n)(*[l.offset for l in d.layers])
        act = _lib.VN_ACT_TANH if wl.activation == "tanh" else _lib.VN_ACT_NONE
        kind = _lib.VN_NOISE_GAUSSIAN if noise == "gaussian" else _lib.VN_NOISE_UNIFORM
        args = (P(d.x.data_ptr()), dt[d.x.dtype], 0, n, c_dims, c_w, c_b, c_off, P(d.seeds.data_ptr()),
                pop, batch, float(wl.sigma), act, kind, P(y.data_ptr()), s)
        el = pop * sum(l.out_f * l.in_f for l in d.layers)
        hbm = (d.x.numel() * d.x.element_size() + y.numel() * 4
               + sum(l.weight.numel() * 4 + l.bias.numel() * 4 for l in d.layers))
        launches.append(Launch("linear_mlp" + suffix, lib.vn_perturbed_mlp_ex, args, el,
                               flops=2.0 * el * batch, hbm_bytes=hbm))
        outputs.append(y)
    elif wl.forward:
        h = d.x
        bufs["x"] = d.x
        for li, l in enumerate(d.layers):
            act = _lib.VN_ACT_TANH if (wl.activation == "tanh" and li < len(d.layers) - 1) else _lib.VN_ACT_NONE
            ydt = torch.bfloat16 if (h.dtype == torch.bfloat16 and l.weight.dtype == torch.bfloat16) else torch.float32
            y = torch.empty((pop, batch, l.out_f), dtype=ydt, device=dev)
            bufs[f"w{li}"], bufs[f"b{li}"] = l.weight, l.bias
            path = lib.vn_perturbed_linear_path(P(h.data_ptr()), dt[h.dtype], 0, P(l.weight.data_ptr()),
                                                dt[l.weight.dtype], batch, l.in_f, l.out_f)
            kernel = ("linear_tc" if path == _lib.VN_PATH_TC else "linear_ffma") + suffix
            args = (P(h.data_ptr()), dt[h.dtype], 0, P(l.weight.data_ptr()), dt[l.weight.dtype],
                    P(l.bias.data_ptr()), dt[l.bias.dtype], P(d.seeds.data_ptr()), pop, batch,
                    l.in_f, l.out_f, float(wl.sigma), l.offset, P(y.data_ptr()), dt[ydt],
                    _lib.VN_PATH_AUTO, act,
                    _lib.VN_NOISE_GAUSSIAN if noise == "gaussian" else _lib.VN_NOISE_UNIFORM, s)
            el = pop * l.out_f * l.in_f
            hbm = h.numel() * h.element_size() + y.numel() * y.element_size() + l.weight.numel() * l.weight.element_size()
            launches.append(Launch(kernel, lib.vn_perturbed_linear_kind, args, el,
                                   flops=2.0 * el * batch, hbm_bytes=hbm))
            h = y
        outputs.append(h)

    # Fitness shaping: the returns' centered ranks, computed on the device, feed
    # the gradient (workloads whose fitness is given as-is use it directly).
    fit = d.fitness
    if wl.grads and d.returns is not None:
        bufs["returns"] = d.returns
        fit = torch.empty_like(d.returns)
        launches.append(Launch("es_ranks", lib.vn_centered_ranks,
                               (P(d.returns.data_ptr()), pop, P(fit.data_ptr()), s), 0,
                               hbm_bytes=pop * 8))
    elif wl.grads:
        bufs["fitness"] = d.fitness
    if flat:
        # The blocks (weights then bias, layer by layer) are laid out by
        # compute_offsets, so the gradients of all of them are one flat range of
        # element indices: one reduction over the population gives every block's
        # gradient as a slice (grad_W of layer l = flat[off_l : off_l + out*in]).
        g = torch.empty((n_params,), dtype=torch.float32, device=dev)
        gw_elems = sum(l.out_f * l.in_f for l in wl.layers)
        if theta is not None:
            # The estimate and the ES step on the parameters, theta += lr * grad (lr
            # fixed for the bench), in one launch (vn_gradient_update).
            launches.append(Launch("grad" + suffix, lib.vn_gradient_update,
                                   (P(fit.data_ptr()), P(d.seeds.data_ptr()), pop, n_params,
                                    float(wl.sigma), wl.layers[0].offset,
                                    _lib.VN_NOISE_GAUSSIAN if noise == "gaussian" else _lib.VN_NOISE_UNIFORM,
                                    ES_LR, P(g.data_ptr()), P(theta.data_ptr()), s),
                                   pop * n_params, hbm_bytes=n_params * 12, grad_w_elems=gw_elems))
            outputs += [g, theta]
        else:
            launches.append(Launch("grad", lib.vn_bias_gradient,
                                   (P(fit.data_ptr()), P(d.seeds.data_ptr()), pop, n_params,
                                    float(wl.sigma), wl.layers[0].offset, P(g.data_ptr()), s),
                                   pop * n_params, hbm_bytes=g.numel() * 4, grad_w_elems=gw_elems))
            outputs.append(g)
    for li, l in enumerate(d.layers if (wl.grads and not flat and noise == "gaussian") else []):
        # The Gaussian-noise variant: the same flat ranges (weights row-major, then
        # the bias block) through the noise-kind entry point.
        gw = torch.empty((l.out_f, l.in_f), dtype=torch.float32, device=dev)
        gb = torch.empty((l.out_f,), dtype=torch.float32, device=dev)
        for blk, n_el, off in ((gw, l.out_f * l.in_f, l.offset), (gb, l.out_f, l.offset + l.out_f * l.in_f)):
            launches.append(Launch("grad_gaussian", lib.vn_gradient_ex,
                                   (P(fit.data_ptr()), P(d.seeds.data_ptr()), pop, n_el, float(wl.sigma),
                                    off, _lib.VN_NOISE_GAUSSIAN, P(blk.data_ptr()), s),
                                   pop * n_el, hbm_bytes=n_el * 4,
                                   grad_w_elems=n_el if blk is gw else 0))
        outputs += [gw, gb]
    for li, l in enumerate(d.layers if (wl.grads and not flat and noise != "gaussian") else []):
        gw = torch.empty((l.out_f, l.in_f), dtype=torch.float32, device=dev)
        gb = torch.empty((l.out_f,), dtype=torch.float32, device=dev)
        launches.append(Launch("grad", lib.vn_weight_gradient,
                               (P(fit.data_ptr()), P(d.seeds.data_ptr()), pop, l.out_f, l.in_f,
                                float(wl.sigma), l.offset, P(gw.data_ptr()), s),
                               pop * l.out_f * l.in_f, hbm_bytes=gw.numel() * 4,
                               grad_w_elems=l.out_f * l.in_f))
        launches.append(Launch("grad", lib.vn_bias_gradient,
                               (P(fit.data_ptr()), P(d.seeds.data_ptr()), pop, l.out_f,
                                float(wl.sigma), l.offset + l.out_f * l.in_f, P(gb.data_ptr()), s),
                               pop * l.out_f, hbm_bytes=gb.numel() * 4))
        outputs += [gw, gb]

    if wl.number in (1, 2) and include_dump:
        dump = torch.empty((pop, n_params), dtype=torch.float32, device=dev)
        launches.append(Launch("noise_dump" + suffix, lib.vn_noise_dump_ex,
                               (P(d.seeds.data_ptr()), pop, n_params, wl.layers[0].offset,
                                _lib.VN_NOISE_GAUSSIAN if noise == "gaussian" else _lib.VN_NOISE_UNIFORM,
                                P(dump.data_ptr()), s),
                               pop * n_params, hbm_bytes=dump.numel() * 4))
        outputs.append(dump)
    return launches, bufs, outputs


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# Distributed plumbing (one process per GPU; rank 0 reports)
# ---------------------------------------------------------------------------

def gpu_id(dev) -> str:
    """nvidia-smi's name for the torch device (PCI bus id; independent of CUDA_VISIBLE_DEVICES)."""
    import torch
    p = torch.cuda.get_device_properties(dev)
    try:
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except AttributeError:
        return "0"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The maximum of ``value`` over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def roofline_of(per_kernel, pk, workload):
    """The roofline object of the dominant kernel (the one with the most time) from the
    kernel pass's per-kernel sums {"ms", "launches", "elements", "flops", "hbm_bytes"}:
    achieved = algorithmic work of its launches / their event time, against each bound
    that applies -- the integer ALU pipe (12 operations per noise element; 13 for the
    Gaussian kind, which also has the MUFU and issue bounds), HBM when the launch has
    algorithmic bytes, the tensor pipe when it has flops -- and the tightest one reported."""
    dom = max(per_kernel, key=lambda n: per_kernel[n]["ms"])
    r = per_kernel[dom]
    secs = r["ms"] * 1e-3
    gaussian = dom.endswith("_gaussian")
    alu_ops = ALU_OPS_GAUSSIAN if gaussian else ALU_OPS_PER_ELEMENT
    cands = {"alu": (r["elements"] * alu_ops / secs / 1e12, pk["alu_ops"] / 1e12, "Tops/s")}
    if gaussian:
        cands["mufu"] = (r["elements"] * MUFU_OPS_GAUSSIAN / secs / 1e12,
                         SMS_NOMINAL * MUFU_LANES_PER_SM * SM_CLOCK_MAX_HZ / 1e12, "Tops/s")
        cands["issue"] = (r["elements"] * OPS_GAUSSIAN / secs / 1e12, pk["issue_ops"] / 1e12, "Tops/s")
    if r["hbm_bytes"]:
        cands["hbm"] = (r["hbm_bytes"] / secs / 1e9, pk["hbm_gbs"], "GB/s")
    if r["flops"]:
        cands["tensor"] = (r["flops"] / secs / 1e12, pk["bf16_tflops"], "TFLOP/s")
    bound = max(cands, key=lambda b: cands[b][0] / cands[b][1])
    ach, peak, unit = cands[bound]
    return {"bound": bound, "kernel": dom, "achieved": ach, "peak": peak, "unit": unit,
            "frac": ach / peak, "traffic": traffic_for(dom, workload),
            "peak_source": ("derived: 152 SMs x 64 integer-ALU lanes x 2.07 GHz" if bound == "alu"
                            else "derived: 152 SMs x 32 MUFU lanes x 2.07 GHz" if bound == "mufu"
                            else "derived: 152 SMs x 128 issue lanes x 2.07 GHz" if bound == "issue"
                            else pk["source"]),
            "ops_per_element": {"alu": alu_ops, "mufu": MUFU_OPS_GAUSSIAN, "issue": OPS_GAUSSIAN}.get(bound),
            # every operation of the element (21, or 32 for the Gaussian variant)
            # through the issue port (152 SMs x 128 lanes x 2.07 GHz)
            "issue_frac": r["elements"] * (OPS_GAUSSIAN if gaussian else OPS_PER_ELEMENT) / secs
                          / pk["issue_ops"],
            "launches": r["launches"], "avg_launch_us": 1e3 * r["ms"] / r["launches"]}


def traffic_for(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel on this
    workload, if the kernel's source is unchanged since the capture (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(f"{kernel}@{workload}")
    if not rec:
        return None
    src = os.path.join(ROOT, "virtual_noise_perturbed_gb300", "csrc", rec["source"])
    if not os.path.exists(src):
        return None
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return rec["bytes_per_launch"] if h == rec["source_sha256_16"] else None


# ---------------------------------------------------------------------------
# The oracle leg (cpu_baseline and --impl reference): the oracle as it stands.
# Each individual's pass is independent of the others', so a sample of
# individuals is split over one spawned process per host core (spawned, not
# forked: the parent has used CUDA). Only the split is parallel; every worker runs
# the oracle's own functions, unchanged, on its individuals.
# ---------------------------------------------------------------------------

def oracle_cores() -> int:
    """The host cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover -- not Linux
        return max(1, os.cpu_count() or 1)


_ORACLE_STATIC = None


def _oracle_init(static):
    """Worker start-up: keep the workload's shared arrays and import the oracle once."""
    global _ORACLE_STATIC
    _ORACLE_STATIC = static
    import oracle.es  # noqa: F401


def _oracle_ready(_):
    return os.getpid()


def _oracle_job(job) -> int:
    """One worker's share of an oracle pass: forward, gradient sums, parameter update
    and noise dump over the individuals whose X rows, seeds and fitness ``job``
    carries. Returns the noise elements regenerated."""
    import numpy as np
    from oracle import es

    st = _ORACLE_STATIC
    x, seeds, fit = job
    k = int(seeds.shape[0])
    if k == 0:
        return 0
    noise, sigma, layers = st["noise"], st["sigma"], st["layers"]
    n = 0
    if st["forward"]:
        h = x.astype(np.float64)
        for li, (w, b, off, in_f, out_f) in enumerate(layers):
            h = es.perturbed_linear(h, w, b, seeds, sigma, off, noise=noise)
            if st["activation"] == "tanh" and li < len(layers) - 1:
                h = np.tanh(h)
            n += k * out_f * in_f
    if st["grads"]:
        for (w, b, off, in_f, out_f) in layers:
            if noise == "gaussian":
                es.gaussian_flat_gradient(fit, seeds, out_f * in_f, sigma, k, off)
                es.gaussian_flat_gradient(fit, seeds, out_f, sigma, k, off + out_f * in_f)
            else:
                gw = es.weight_gradient(fit, seeds, (out_f, in_f), sigma, k, off)
                gb = es.bias_gradient(fit, seeds, (out_f,), sigma, k, off + out_f * in_f)
                if st["update"]:
                    es.es_update(w, gw, ES_LR)
                    es.es_update(b, gb, ES_LR)
            n += k * (out_f * in_f + out_f)
    if st["dump_n"]:
        (es.gaussian_dump if noise == "gaussian" else es.noise_dump)(seeds, st["dump_n"], st["dump_offset"])
        n += k * st["dump_n"]
    return n


class OraclePool:
    """The oracle's pass over sampled individuals of ``wl``, on ``cores`` spawned workers."""

    def __init__(self, wl, noise: str = "uniform", cores: int = None):
        import multiprocessing as mp

        self.wl, self.noise = wl, noise
        self.cores = cores or oracle_cores()
        n_params = sum(l.out_f * l.in_f + l.out_f for l in wl.layers)
        static = {
            "noise": noise, "sigma": wl.sigma, "activation": wl.activation,
            "forward": wl.forward, "grads": wl.grads,
            "update": wl.forward and wl.grads and len(wl.layers) > 1,
            "dump_n": n_params if wl.number in (1, 2) else 0,
            "dump_offset": wl.layers[0].offset,
            "layers": [(l.weight.float().numpy(), None if l.bias is None else l.bias.float().numpy(),
                        l.offset, l.in_f, l.out_f) for l in wl.layers],
        }
        self.x = wl.x.float().numpy() if wl.forward else None
        self.seeds = wl.seeds.numpy()
        ctx = mp.get_context("spawn")
        self.pool = ctx.Pool(self.cores, initializer=_oracle_init, initargs=(static,))
        self.pool.map(_oracle_ready, range(self.cores), chunksize=1)  # every worker up and importing

    def run(self, individuals: int):
        """One pass over the first ``individuals`` individuals: the fitness (the centered
        ranks of the whole population's returns, where the workload shapes them; a
        rank is global), then the individuals split evenly over the workers.
        Returns (noise elements, seconds)."""
        import numpy as np
        from oracle import es

        t0 = time.monotonic()
        wl = self.wl
        if wl.grads and wl.returns is not None:
            fit = es.centered_ranks(wl.returns.numpy())
        else:
            fit = wl.fitness.numpy()
        parts = [p for p in np.array_split(np.arange(individuals), self.cores) if p.size]
        jobs = [(None if self.x is None else self.x[p], self.seeds[p], fit[p]) for p in parts]
        n = sum(self.pool.map(_oracle_job, jobs, chunksize=1))
        return n, time.monotonic() - t0

    def calibrate(self, budget_s: float) -> int:
        """Individuals of one pass that take about ``budget_s`` (one per core first)."""
        one = min(self.wl.pop, self.cores)
        _, t = self.run(one)
        per_round = max(t, 1e-3)
        rounds = max(1, int(budget_s / per_round))
        return int(min(self.wl.pop, one * rounds))

    def close(self):
        self.pool.close()
        self.pool.join()


def sample_text(wl, inds: int, cores: int) -> str:
    parts = ["forward"] if wl.forward else []
    if wl.grads:
        parts.append("gradient sums")
    if wl.number in (1, 2):
        parts.append("noise dump")
    return (f"the oracle's pass ({', '.join(parts)}) over the first {inds} of {wl.pop} individuals, "
            f"split over {cores} spawned processes (one per host core)")


def time_oracle(wl, budget_s: float, noise: str = "uniform"):
    """The cpu_baseline: one oracle pass on all host cores over as many individuals as
    fit about ``budget_s``. Returns (elements/s, individuals, seconds, cores)."""
    pool = OraclePool(wl, noise)
    try:
        inds = pool.calibrate(budget_s)
        n, t = pool.run(inds)
    finally:
        pool.close()
    return n / t, inds, t, pool.cores


# ---------------------------------------------------------------------------

def step_elements(wl, include_dump: bool = True) -> int:
    """Noise elements one step of ``wl`` regenerates (forward, gradients, dump), as
    ``build_step`` counts them: pop x weights for the forward, pop x parameters for
    the gradients and for the dump of the ES workloads."""
    n_params = sum(l.out_f * l.in_f + l.out_f for l in wl.layers)
    el = wl.pop * sum(l.out_f * l.in_f for l in wl.layers) if wl.forward else 0
    if wl.grads:
        el += wl.pop * n_params
    if wl.number in (1, 2) and include_dump:
        el += wl.pop * n_params
    return el


def compute_dtype(wl) -> str:
    """The arithmetic type of the step's contraction: bf16 where the forward runs on
    the tensor cores (bf16 activations), f32 otherwise (the policy chain, the CUDA-core
    forward, and the gradient-only step, which has no forward)."""
    import torch
    return "bf16" if wl.forward and wl.x.dtype == torch.bfloat16 else "f32"


def config_for(wl, world, noise="uniform"):
    return {"workload": wl.name, "description": wl.description, "noise": noise, "pop": wl.pop, "batch": wl.batch,
            "layers": [[l.in_f, l.out_f] for l in wl.layers], "sigma": wl.sigma,
            "noise_elements_per_step": step_elements(wl), "l2": "256 MiB buffer rewritten between timed steps",
            "parallelism": f"population shards x{world} (independent per rank)"}


def run_reference(args, wl, world, rank):
    """The oracle alone, as it stands, on the host's cores: W warm-up passes, then K
    timed passes, each over a bounded sample of the workload's individuals."""
    if rank != 0:
        return 0
    budget = min(4.0, 100.0 / max(1, args.steps))
    pool = OraclePool(wl, args.noise)
    try:
        one = min(wl.pop, pool.cores)
        for _ in range(args.warmup):
            _, t_one = pool.run(one)
        inds = int(min(wl.pop, one * max(1, int(budget / max(t_one, 1e-3)))))
        total_el, total_t = 0, 0.0
        for _ in range(args.steps):
            n, t = pool.run(inds)
            total_el += n
            total_t += t
    finally:
        pool.close()
    rate = total_el / total_t
    cfg = config_for(wl, 1, args.noise)
    line = {"metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
            "impl": "reference",
            "cpu_baseline": {"value": rate, "unit": UNIT, "cores": pool.cores, "kind": "oracle",
                             "sample": "each step: " + sample_text(wl, inds, pool.cores)},
            "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU measurement of one workload
# ---------------------------------------------------------------------------

def measure(wl, dev, stream, flush, args, world, noise, steps=None, include_dump=True):
    """Warm-up, the step pass and the kernel pass of one workload on this rank.

    ``steps`` None: exactly --steps steps (the headline); else at most that many,
    as many as fit --extra-seconds by the last warm-up step's time (at least 3)."""
    import torch

    launches, bufs, outputs = build_step(wl, dev, stream.cuda_stream, noise, include_dump)
    res = {"n_launches": len(launches), "el_step": sum(l.elements for l in launches)}
    with torch.cuda.stream(stream):
        wa, wb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for w in range(args.warmup):
            if w == args.warmup - 1:
                wa.record(stream)
            for l in launches:
                l()
            if w == args.warmup - 1:
                wb.record(stream)
            flush.zero_()
        torch.cuda.synchronize(dev)
        est_ms = max(wa.elapsed_time(wb), 1e-3)
        if steps is None:
            k_steps = args.steps
            k_kern = args.kernel_steps if args.kernel_steps is not None else args.steps
        else:
            k_steps = k_kern = int(min(args.steps, max(3, args.extra_seconds * 1e3 / est_ms)))
        # The step pass replays the step's C-ABI calls captured once as a CUDA graph
        # (the same kernels and arguments; the graph only removes the host launch
        # latency between them). If capture is refused, the calls are made directly.
        graph, graph_error = None, None
        if not args.no_graph:
            try:
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=stream):
                    for l in launches:
                        l()
                graph.replay()
                torch.cuda.synchronize(dev)
            except Exception as exc:  # noqa: BLE001 -- reported in the JSON line
                graph = None
                graph_error = f"{type(exc).__name__}: {exc}"[:200]
                torch.cuda.synchronize(dev)
        ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(k_steps)]
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(launches))]
              for _ in range(k_kern)]
        barrier(world)
        torch.cuda.synchronize(dev)
        wall0 = time.perf_counter()
        for k in range(k_steps):
            ev_step[k][0].record(stream)
            if graph is not None:
                graph.replay()
            else:
                for l in launches:
                    l()
            ev_step[k][1].record(stream)
            flush.zero_()
        torch.cuda.synchronize(dev)
        res["wall_s"] = time.perf_counter() - wall0
        barrier(world)
        torch.cuda.synchronize(dev)
        for k in range(k_kern):
            for j, l in enumerate(launches):
                ev[k][2 * j].record(stream)
                l()
                ev[k][2 * j + 1].record(stream)
            flush.zero_()
        torch.cuda.synchronize(dev)
        barrier(world)
    per_kernel = {}
    for k in range(k_kern):
        for j, l in enumerate(launches):
            ms = ev[k][2 * j].elapsed_time(ev[k][2 * j + 1])
            rec = per_kernel.setdefault(l.kernel, {"ms": 0.0, "launches": 0, "elements": 0, "flops": 0.0,
                                                   "hbm_bytes": 0.0, "grad_w_elems": 0})
            rec["ms"] += ms
            rec["launches"] += 1
            rec["elements"] += l.elements
            rec["flops"] += l.flops
            rec["hbm_bytes"] += l.hbm_bytes
            rec["grad_w_elems"] += l.grad_w_elems
    total_ms = sum(a.elapsed_time(b) for a, b in ev_step)
    res.update({"steps": k_steps, "kernel_steps": k_kern, "total_ms_max": max_over_ranks(total_ms, world, dev),
                "per_kernel": per_kernel, "graph": graph is not None, "graph_error": graph_error,
                "gpu_launches": len(launches) * (k_steps + k_kern)})
    return res


def summarise(wl, res, world, pk):
    """value, ms per step, the dominant kernel's roofline, per-kernel shares and the
    phase metrics of one measured workload."""
    per_kernel = res["per_kernel"]
    value = res["el_step"] * res["steps"] * world / (res["total_ms_max"] * 1e-3)
    all_ms = sum(x["ms"] for x in per_kernel.values())
    kernels = {n: {"launches": v["launches"], "share": v["ms"] / all_ms, "avg_us": 1e3 * v["ms"] / v["launches"],
                   "noise_elem_per_s": v["elements"] / (v["ms"] * 1e-3)} for n, v in per_kernel.items()}
    fwd = [n for n in per_kernel if n.startswith("linear")]
    grads = [n for n in per_kernel if n.startswith("grad")]
    fwd_ms = sum(per_kernel[n]["ms"] for n in fwd)
    grad_ms = sum(per_kernel[n]["ms"] for n in grads)
    gw = sum(per_kernel[n]["grad_w_elems"] for n in grads)
    return {
        "value": value, "unit": UNIT, "ms_per_step": res["total_ms_max"] / res["steps"],
        "steps": res["steps"], "noise_elements_per_step": res["el_step"],
        "roofline": roofline_of(per_kernel, pk, wl.name),
        "kernels": kernels,
        "perturbed_linear_tflops": (sum(per_kernel[n]["flops"] for n in fwd) / (fwd_ms * 1e-3) / 1e12)
                                   if fwd else None,
        "grad_w_elem_per_s": (gw / (grad_ms * 1e-3)) if grads and gw else None,
        "launch": ("step pass: one CUDA graph of the step's C-ABI calls per step" if res["graph"] else
                   "step pass: direct C-ABI calls" + (f" (graph capture failed: {res['graph_error']})"
                                                      if res["graph_error"] else "")),
    }


def measure_hash_peak(dev, stream, reps: int = 10):
    """The hash-only kernel (vn_hash_probe) on every SM at full occupancy: 2048 threads
    per SM, 4 rounds, 4096 elements per thread. Its element rate x 12 ALU-pipe
    operations per element is the measured ceiling of the integer ALU pipe."""
    import torch
    from virtual_noise_perturbed_gb300 import _lib

    lib = _lib.load()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    n_sums, m = sms * 2048 * 4, 4096
    sums = torch.empty(n_sums, dtype=torch.float32, device=dev)
    args = (0x5EED, 0, n_sums, m, ctypes.c_void_p(sums.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
    with torch.cuda.stream(stream):
        for _ in range(3):
            _lib.check(lib.vn_hash_probe(*args), "vn_hash_probe")
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            a.record(stream)
            _lib.check(lib.vn_hash_probe(*args), "vn_hash_probe")
            b.record(stream)
        torch.cuda.synchronize(dev)
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    el = n_sums * m
    rate = el / (ms * 1e-3)
    return {"kernel": "hash_probe", "elem_per_s": rate, "ops_per_element": ALU_OPS_PER_ELEMENT,
            "tops": rate * ALU_OPS_PER_ELEMENT / 1e12, "ms": ms, "launches": reps,
            "elements_per_launch": el,
            "derived_tops": SMS_NOMINAL * ALU_LANES_PER_SM * SM_CLOCK_MAX_HZ / 1e12,
            "launch": f"{sms} SMs x 2048 threads x 4 rounds, {m} elements per thread; median of {reps}"}


def with_measured_peak(roof, hp):
    """Add the measured ALU ceiling beside an alu-bound roofline's derived peak."""
    if hp is not None and roof.get("bound") == "alu":
        roof["peak_measured"] = hp["tops"]
        roof["frac_of_measured"] = roof["achieved"] / hp["tops"]
        roof["peak_measured_source"] = "measured: vn_hash_probe (the hash alone) in this run"
    return roof


EXTRA_DEFAULT = ["mid", "grad_only", "es_mlp", "tiny"]


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["vn", "reference"], default="vn")
    ap.add_argument("--workload", default="large_tc",
                    choices=["tiny", "es_mlp", "mid", "grad_only", "large_tc"])
    ap.add_argument("--extras", default="auto",
                    help="workloads measured besides the headline: 'auto' (the other four when the "
                         "headline is large_tc, else none), 'none', or a comma-separated list")
    ap.add_argument("--extra-seconds", type=float, default=2.5,
                    help="timed-region budget of each extra workload's step pass")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--no-graph", action="store_true",
                    help="step pass: direct C-ABI calls instead of a CUDA graph of them")
    ap.add_argument("--kernel-steps", type=int, default=None,
                    help="steps of the headline's per-kernel timing pass (default: --steps)")
    ap.add_argument("--pop", type=int, default=None,
                    help="run only the headline workload's first POP individuals (smaller profiling cases)")
    ap.add_argument("--noise", choices=["uniform", "gaussian"], default="uniform",
                    help="gaussian: the Box-Muller noise variant throughout (not on the tiny workload)")
    ap.add_argument("--cpu-baseline-seconds", type=float, default=16.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-hash-peak", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.noise == "gaussian" and args.workload == "tiny":
        ap.error("--noise gaussian applies to the es_mlp, mid, grad_only and large_tc workloads")

    from virtual_noise_perturbed_gb300 import workloads
    numbers = {v: k for k, v in workloads.NAMES.items()}
    if args.extras == "auto":
        extras = [e for e in EXTRA_DEFAULT if e != args.workload] if args.workload == "large_tc" else []
    elif args.extras == "none":
        extras = []
    else:
        extras = [e.strip() for e in args.extras.split(",") if e.strip()]
        bad = [e for e in extras if e not in numbers]
        if bad:
            ap.error(f"unknown workloads in --extras: {bad}")
    if args.noise == "gaussian":
        extras = [e for e in extras if e != "tiny"]
    world, rank, local = dist_env()

    def load(name, pop=None):
        wl = workloads.make(numbers[name])
        if pop is not None:
            wl = wl.first(pop)
        if rank > 0:  # independent population per rank
            wl.seeds = wl.seeds + rank * wl.pop
        return wl

    wl = load(args.workload, args.pop)
    if args.impl == "reference":
        return run_reference(args, wl, world, rank)

    import torch
    if not torch.cuda.is_available():
        print(json.dumps({"metric": METRIC, "error": "no CUDA device"}))
        return 1
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from virtual_noise_perturbed_gb300 import _lib, build as vbuild
    vbuild.build()
    stream = torch.cuda.Stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    pk = peaks()

    sampler = ClockSampler(gpu_id(dev))
    head = measure(wl, dev, stream, flush, args, world, args.noise)
    launches_total = head["gpu_launches"]
    extra_res = {}
    for name in extras:
        xw = load(name)
        r = measure(xw, dev, stream, flush, args, world, args.noise, steps=args.steps)
        extra_res[name] = (xw, r)
        launches_total += r["gpu_launches"]
    hp = None
    if not args.no_hash_peak:
        hp = measure_hash_peak(dev, stream)
        launches_total += hp["launches"]
    clocks = sampler.stop()
    status = _lib.load().vn_device_status(ctypes.c_void_p(stream.cuda_stream))
    if status != 0:
        raise _lib.VNError(status, "bench")

    s_head = summarise(wl, head, world, pk)
    with_measured_peak(s_head["roofline"], hp)
    configs = {}
    for name, (xw, r) in extra_res.items():
        s = summarise(xw, r, world, pk)
        with_measured_peak(s["roofline"], hp)
        s["description"] = xw.description
        s["dtype"] = compute_dtype(xw)
        configs[name] = s

    # --- end to end: host buffers, copies inside the timed region
    e2e = run_e2e(wl, dev, stream, args.e2e_steps, world, head["el_step"], args.noise)
    launches_total += head["n_launches"] * e2e["steps"]
    for name, (xw, r) in extra_res.items():
        steps = int(min(args.e2e_steps, max(3, args.extra_seconds * 1e3 / max(configs[name]["ms_per_step"], 1e-3))))
        configs[name]["e2e"] = run_e2e(xw, dev, stream, steps, world, r["el_step"], args.noise)
        launches_total += r["n_launches"] * steps
        if xw.number in (1, 2):
            # The same step without the noise dump: its 4-byte-per-element copy back
            # dominates the host link, so the forward + ranks + gradient + update
            # step is reported on its own as well.
            el = step_elements(xw, include_dump=False)
            configs[name]["e2e_no_dump"] = run_e2e(xw, dev, stream, steps, world, el, args.noise,
                                                   include_dump=False)
            launches_total += (r["n_launches"] - 1) * steps

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, inds, tt, cores = time_oracle(wl, args.cpu_baseline_seconds, noise=args.noise)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": sample_text(wl, inds, cores) + f", {tt:.1f} s"}

    if rank == 0:
        cfg = config_for(wl, world, args.noise)
        cfg["noise_elements_per_step"] = head["el_step"]
        cfg["launch"] = s_head["launch"]
        line = {"metric": METRIC, "value": s_head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": s_head["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": compute_dtype(wl),
                "data": "synthetic", "config": cfg, "roofline": s_head["roofline"], "cpu_baseline": cpu,
                "e2e": e2e, "gpu_launches": launches_total, "clocks": clocks,
                "kernels": s_head["kernels"],
                "perturbed_linear_tflops": s_head["perturbed_linear_tflops"],
                "grad_w_elem_per_s": s_head["grad_w_elem_per_s"],
                "noise_elements_per_step": head["el_step"],
                "configs": configs, "alu_peak_measured": hp,
                "wall_s_timed_region": head["wall_s"]}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_e2e(wl, dev, stream, steps, world, el_step, noise, include_dump=True):
    """The same step through the C ABI with inputs in pinned host memory: each step
    copies its inputs host -> device, runs, and copies every result back.

    Three sets of device buffers rotate between steps, and the copies run on
    streams of their own, so that step k+1's host->device copy and step k-1's
    device->host copy overlap step k's kernels (the two copy directions use
    separate engines). A set's inputs are rewritten only after the kernels that
    read them have finished, and its outputs only after they have reached the host;
    with three sets that waits on step k-2, so neither copy direction has to wait for
    the other (with two, step k+1's inputs would wait for step k-1's results to reach
    the host)."""
    import torch
    copy_stream = torch.cuda.Stream(dev)   # device -> host
    load_stream = torch.cuda.Stream(dev)   # host -> device
    sets = []
    for _ in range(E2E_SETS):
        launches, bufs, outputs = build_step(wl, dev, stream.cuda_stream, noise, include_dump)
        sets.append((launches, bufs, outputs))
    host_in = {k: v.detach().cpu().pin_memory() for k, v in sets[0][1].items()
               if v is not None and v.numel()}
    host_out = [[o.detach().cpu().pin_memory() for o in st[2]] for st in sets]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out[0])
    loaded = [torch.cuda.Event() for _ in sets]
    computed = [torch.cuda.Event() for _ in sets]
    copied = [torch.cuda.Event() for _ in sets]

    def one(k):
        j = k % E2E_SETS
        launches, bufs, outputs = sets[j]
        with torch.cuda.stream(load_stream):
            load_stream.wait_event(computed[j])   # the kernels that read this set are done
            load_stream.wait_event(copied[j])     # and its results (theta is both) are out
            for name, v in host_in.items():
                bufs[name].copy_(v, non_blocking=True)
            loaded[j].record(load_stream)
        with torch.cuda.stream(stream):
            stream.wait_event(loaded[j])
            stream.wait_event(copied[j])          # this set's last results are on the host
            for l in launches:
                l()
            computed[j].record(stream)
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(computed[j])
            for o, h in zip(outputs, host_out[j]):
                h.copy_(o, non_blocking=True)
            copied[j].record(copy_stream)

    for e in computed:
        e.record(stream)
    for c in copied:
        c.record(copy_stream)
    for k in range(E2E_SETS):
        one(k)
    torch.cuda.synchronize(dev)
    barrier(world)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    load_stream.wait_stream(stream)
    copy_stream.wait_stream(stream)
    for k in range(steps):
        one(k)
    stream.wait_stream(copy_stream)
    stream.wait_stream(load_stream)
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(a.elapsed_time(b), world, dev)
    link = host_link(sets[0], host_in, host_out[0], load_stream, copy_stream, dev)
    link["frac"] = link["bound_ms_per_step"] / (ms / steps)
    return {"value": el_step * steps * world / (ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": ms / steps,
            "copies": f"step k+1's inputs copied in and step k-1's results copied back on streams "
                      f"of their own while step k runs ({E2E_SETS} rotating buffer sets)", "host_link": link}


def host_link(step_set, host_in, host_out, load_stream, copy_stream, dev, reps=5):
    """The host link's own floor for one e2e step: the step's input copies alone and its
    result copies alone, each timed with events on its own stream (the two directions
    run on separate copy engines, so a pipelined step can take no less than the slower)."""
    import torch
    _, bufs, outputs = step_set

    def timed(stream, body):
        body()
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            body()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / reps

    def load():
        with torch.cuda.stream(load_stream):
            for name, v in host_in.items():
                bufs[name].copy_(v, non_blocking=True)

    def back():
        with torch.cuda.stream(copy_stream):
            for o, h in zip(outputs, host_out):
                h.copy_(o, non_blocking=True)

    h2d_ms = timed(load_stream, load)
    d2h_ms = timed(copy_stream, back)
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out)
    def gbs(nbytes, ms):
        return nbytes / (ms * 1e-3) / 1e9 if ms > 0 else None

    return {"h2d_ms": h2d_ms, "d2h_ms": d2h_ms, "h2d_gbs": gbs(h2d, h2d_ms), "d2h_gbs": gbs(d2h, d2h_ms),
            "bound_ms_per_step": max(h2d_ms, d2h_ms)}


if __name__ == "__main__":
    sys.exit(main())
