"""Benchmark of the routed-expert block-quantized MoE FFN on GB300 (libftmoe).

Default workload: the largest single-GPU configuration -- FP8 prefill, 4,096 tokens routed
top-6 over 256 experts (24,576 routes, about 96 rows per expert), hidden 7168, per-expert
intermediate 2048, FP8-e4m3 weights with 128x128 fp32 block scales -- replayed from one CUDA
graph while the routes and inputs change between steps. A step is one ftmoe_moe_forward
(quantize + segment -> gather -> gate/up -> SiLU-and-mul -> down -> combine). The decode,
gather and NVFP4 workloads are selected with --workload.

Timing: W warm-up steps, then K timed steps; before every step the inputs of the
next route set are copied into the graph's input buffers and L2 is flushed (a 512 MiB
write, then a 256 MiB read that writes the flush's dirty lines back), both outside the
timed events; each step is bracketed by CUDA events on the
launching stream; barrier + synchronize on both sides of the timed loop; max over
ranks. `value` is microseconds per call for the whole job (time / calls of all ranks).

Prints one JSON line. --impl reference times the CPU oracle instead (host cores).
"""
import argparse
import json
import os
import subprocess
import sys
import time

# the CPU oracle legs use one BLAS thread so the reported core count is exact
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

WORKLOADS = {
    # name: (tokens, hidden, inter, experts, topk, active per token,
    #        path: 0 automatic, 1 route slots (streaming kernel), 2 grouped (tcgen05) with the
    #        separate SiLU-and-mul kernel, 3 grouped with SiLU-and-mul fused into gate/up)
    "decode-h4096-i1024-e64-t8-a8": (8, 4096, 1024, 64, 8, 8, 0),
    "decode-h4096-i1024-e64-t1-a8": (1, 4096, 1024, 64, 8, 8, 0),
    "decode-h4096-i1024-e64-t8-a4": (8, 4096, 1024, 64, 8, 4, 0),
    "decode-h4096-i1024-e64-t8-a2": (8, 4096, 1024, 64, 8, 2, 0),
    "decode-h4096-i1024-e64-t8-a0": (8, 4096, 1024, 64, 8, 0, 0),
    "decode-h4096-i1024-e64-t1-a4": (1, 4096, 1024, 64, 8, 4, 0),
    "decode-h4096-i1024-e64-t1-a2": (1, 4096, 1024, 64, 8, 2, 0),
    "decode-h4096-i1024-e64-t1-a0": (1, 4096, 1024, 64, 8, 0, 0),
    "decode-h2048-i768-e8-t1-a2": (1, 2048, 768, 8, 8, 2, 0),
    # one path forced, to compare them
    "decode-h4096-i1024-e64-t8-a8-slots": (8, 4096, 1024, 64, 8, 8, 1),
    "decode-h4096-i1024-e64-t1-a8-slots": (1, 4096, 1024, 64, 8, 8, 1),
    "decode-h4096-i1024-e64-t1-a2-slots": (1, 4096, 1024, 64, 8, 2, 1),
    "decode-h2048-i768-e8-t1-a2-slots": (1, 2048, 768, 8, 8, 2, 1),
    "decode-h4096-i1024-e64-t2-a8": (2, 4096, 1024, 64, 8, 8, 0),
    "decode-h4096-i1024-e64-t2-a8-slots": (2, 4096, 1024, 64, 8, 8, 1),
    "decode-h4096-i1024-e64-t8-a8-sep": (8, 4096, 1024, 64, 8, 8, 2),
    # path 4: the fused decode kernel (gate/up, SiLU-and-mul, down and combine in one launch)
    **{f"decode-h4096-i1024-e64-t{t}-a{a}-dk": (t, 4096, 1024, 64, 8, a, 4) for t in (1, 8) for a in (8, 4, 2, 0)},
    "decode-h2048-i768-e8-t1-a2-dk": (1, 2048, 768, 8, 8, 2, 4),
    "prefill-fp8-h7168-i2048-e256-r1536": (256, 7168, 2048, 256, 6, 6, 0),
    "prefill-fp8-h7168-i2048-e256-r6144": (1024, 7168, 2048, 256, 6, 6, 0),
    "prefill-fp8-h7168-i2048-e256-r24576": (4096, 7168, 2048, 256, 6, 6, 0),
    "prefill-fp8-h7168-i2048-e256-r1536-sep": (256, 7168, 2048, 256, 6, 6, 2),
    "prefill-fp8-h7168-i2048-e256-r6144-sep": (1024, 7168, 2048, 256, 6, 6, 2),
    "prefill-fp8-h7168-i2048-e256-r24576-sep": (4096, 7168, 2048, 256, 6, 6, 2),
    "prefill-fp8-h7168-i2048-e256-r24576-comb": (4096, 7168, 2048, 256, 6, 6, 5),
    # a 32-expert bank with the same rows per expert (96) as the 24,576-route case: small
    # enough (1.4 GB of weights) for multi-pass profiler captures
    "prefill-fp8-h7168-i2048-e32-r3072": (512, 7168, 2048, 32, 6, 6, 0),
    "prefill-fp8-h7168-i2048-e32-r3072-sep": (512, 7168, 2048, 32, 6, 6, 2),
    # NVFP4 weights and activations (e2m1, one e4m3 scale per 16 elements, fp32 tensor
    # scales) on the same prefill geometry
    "prefill-nvfp4-h7168-i2048-e256-r6144": (1024, 7168, 2048, 256, 6, 6, 2),
    "prefill-nvfp4-h7168-i2048-e256-r24576": (4096, 7168, 2048, 256, 6, 6, 2),
    "prefill-nvfp4-h7168-i2048-e32-r3072": (512, 7168, 2048, 32, 6, 6, 2),
    # MXFP8 (e4m3 codes, one E8M0 scale per 32 elements; the bf16 activation is gathered and
    # quantized after the gather): the prefill geometry
    "prefill-mxfp8-h7168-i2048-e256-r6144": (1024, 7168, 2048, 256, 6, 6, 2),
    "prefill-mxfp8-h7168-i2048-e256-r24576": (4096, 7168, 2048, 256, 6, 6, 2),
    "prefill-mxfp8-h7168-i2048-e32-r3072": (512, 7168, 2048, 32, 6, 6, 2),
}
DEFAULT_WORKLOAD = "prefill-fp8-h7168-i2048-e256-r24576"

# The fused FP8 row + scale gather alone: name -> (k, tokens, top-k). Source rows are random
# FP8 bytes [tokens x k] with fp32 scales U(1e-3, 1) per 128 columns; the map has
# tokens * top-k entries drawn by randint over [0, tokens) (duplicates expected).
GATHER_WORKLOADS = {f"gather-k{k}-t{t}": (k, t, 8) for k in (7168, 2048, 896) for t in (1, 8, 64, 1024)}


# The pages' own per-call times for exactly these workloads (other GPUs: context, not a
# target), so that vs_baseline = value / page value (below 1 = faster):
# - FreeToken "perf(moe): skip inactive block-fp8 decode routes", GPU decode A/B table:
#   RTX A1000 (sm_86, its FP8 compatibility path), batch 1, top-k 8, CUDA graphs;
# - SGLang "Gather the cutlass MoE activation and its scales in one launch", Speed Tests:
#   the fused gather on B200, top-k 8.
PAGES_US = {
    "decode-h2048-i768-e8-t1-a2": 60.589,
    "decode-h4096-i1024-e64-t1-a8": 472.730,
    "decode-h4096-i1024-e64-t1-a4": 255.034,
    "decode-h4096-i1024-e64-t1-a2": 148.278,
    "decode-h4096-i1024-e64-t1-a0": 8.819,
    "gather-k7168-t1": 1.31,
    "gather-k2048-t1": 1.42,
    "gather-k7168-t8": 1.60,
    "gather-k7168-t64": 2.10,
    "gather-k7168-t1024": 11.14,
}


def vs_pages(workload, value_us):
    # the same workload on another forward path of this library has the same page number
    ref = PAGES_US.get(workload[:-3] if workload.endswith("-dk") else workload)
    return None if ref is None else round(value_us / ref, 4)


def workload_format(name):
    return "nvfp4" if "-nvfp4-" in name else ("mxfp8" if "-mxfp8-" in name else "fp8")


def code_bytes(fmt, n):
    """Bytes of one quantized row of n elements."""
    return n // 2 if fmt == "nvfp4" else n


def scale_bytes(fmt, n):
    """Bytes of the scales of one quantized activation row of n elements."""
    if fmt == "mxfp8":
        return n // 32
    return 4 * (-(-n // 128)) if fmt == "fp8" else n // 16


def weight_bytes(fmt, n, k):
    """Bytes of one expert matrix [n, k] with its scales."""
    if fmt == "fp8":
        return n * k + 4 * (-(-n // 128)) * (-(-k // 128))
    if fmt == "mxfp8":
        return n * k + n * k // 32
    return n * k // 2 + n * k // 16 + 4


def code_hash(path):
    """First 12 hex digits of the sha1 of a C/C++/CUDA source's code: // and /* */ comments,
    trailing blanks and blank lines removed. Editing a comment keeps a recorded capture
    valid; any change to the code voids it."""
    import hashlib
    text = open(path).read()
    out, i, n, quote = [], 0, len(text), None
    while i < n:
        c = text[i]
        if quote:
            out.append(c)
            if c == "\\" and i + 1 < n:
                out.append(text[i + 1])
                i += 2
                continue
            if c == quote:
                quote = None
            i += 1
        elif c in "\"'":
            quote = c
            out.append(c)
            i += 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = [ln.rstrip() for ln in "".join(out).splitlines()]
    return hashlib.sha1("\n".join(ln for ln in lines if ln).encode()).hexdigest()[:12]


def recorded_traffic(workload):
    """DRAM bytes per launch of the dominant kernel from profiles/traffic.txt, or None when
    no capture is recorded or the kernel's code changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    for ln in open(path):
        parts = ln.split()
        if len(parts) != 4 or ln.startswith("#") or parts[0] != workload:
            continue
        src = os.path.join(ROOT, "block_quantized_moe_gb300", parts[1])
        if not os.path.exists(src):
            return None
        return int(parts[3]) if code_hash(src) == parts[2] else None
    return None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ------------------------------------------------------------------------------------
# distributed plumbing (replicas: each rank runs its own copy of the workload)
# ------------------------------------------------------------------------------------

def dist_init(backend=None):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, device):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ------------------------------------------------------------------------------------

class ClockSampler:
    """SM clock and clock-event reasons during the timed region.

    Sampled about every millisecond from a thread through NVML (libnvidia-ml via ctypes,
    read-only queries), so that even a region of a few milliseconds gets samples; falls
    back to `nvidia-smi -lms 50` when NVML cannot be loaded."""
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        import ctypes
        self.ct = ctypes
        self.device = device
        self.samples = []
        self.thread = None
        self.proc = None
        self.nv = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            pr = torch.cuda.get_device_properties(device)
            bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle for " + bus)
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) != 0:  # 1 = SM clock
                raise OSError("max clock query failed")
            self.reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None)
            if self.reasons_fn is None:
                self.reasons_fn = nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.nv, self.h, self.max_mhz = nv, h, float(mx.value)
        except (OSError, AttributeError):
            self.nv = None

    @classmethod
    def summarize(cls, samples, max_mhz):
        """(sm MHz, reason bit mask) samples -> the bench line's clocks object."""
        if not samples:
            return None
        reasons = sorted({name for _, r in samples for bit, name in cls.REASON_BITS.items() if r & bit})
        return {"sm_mhz": float(np.median([c for c, _ in samples])), "sm_max_mhz": max_mhz,
                "reasons": reasons, "samples": len(samples), "source": "nvml"}

    def _poll(self):
        ct = self.ct
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        while not self.stop_flag:
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(clk)) == 0 and \
                    self.reasons_fn(self.h, ct.byref(rs)) == 0:
                self.samples.append((float(clk.value), int(rs.value)))
            time.sleep(0.001)

    def start(self):
        if self.nv is not None:
            import threading
            self.stop_flag = False
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix=f"clocks_dev{self.device.index or 0}_", suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.device.index or 0),
                                          f"--query-gpu={self.SMI_FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.thread is not None:
            self.stop_flag = True
            self.thread.join(timeout=5)
            return self.summarize(self.samples, self.max_mhz)
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            lines = fh.readlines()
        os.unlink(self.path)
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi"}


# ------------------------------------------------------------------------------------
# workload construction (inputs resident in HBM before timing starts)
# ------------------------------------------------------------------------------------

class MoeWorkload:
    NSETS = 8  # route/input sets rotated between steps (2 for the prefill sizes)

    def __init__(self, name, device, seed=0xF7E00002):
        import block_quantized_moe_gb300 as ft
        self.ft = ft
        T, H, I, E, k, active, path = WORKLOADS[name]
        self.name, self.T, self.H, self.I, self.E, self.k, self.active, self.path = name, T, H, I, E, k, active, path
        self.dev = device
        if T >= 256:
            self.NSETS = 2
        self.fmt = workload_format(name)
        self.ft_fmt = {"fp8": ft.FMT_FP8, "nvfp4": ft.FMT_NVFP4, "mxfp8": ft.FMT_MXFP8}[self.fmt]
        banks = []
        for n, kk, tag in ((2 * I, H, "gateup"), (H, I, "down")):
            if self.fmt == "fp8":
                q = torch.empty(E, n, kk, dtype=torch.uint8, device=device)
                sc = torch.empty(E, -(-n // 128), -(-kk // 128), dtype=torch.float32, device=device)
                gsc = None
            elif self.fmt == "mxfp8":
                q = torch.empty(E, n, kk, dtype=torch.uint8, device=device)
                sc = torch.empty(E, n, kk // 32, dtype=torch.uint8, device=device)
                gsc = None
            else:
                q = torch.empty(E, n, kk // 2, dtype=torch.uint8, device=device)
                sc = torch.empty(E, n, kk // 16, dtype=torch.uint8, device=device)
                gsc = torch.empty(E, dtype=torch.float32, device=device)
            for e in range(E):
                ft.ftmoe_quantize_weights(synth.expert_weight_fp32(n, kk, seed, e, tag, device)[None],
                                          q[e:e + 1], sc[e:e + 1], None if gsc is None else gsc[e:e + 1],
                                          fmt=self.ft_fmt)
            banks.append((q, sc, gsc))
        self._banks = banks
        self.bank_gu = ft.make_bank(*banks[0], fmt=self.ft_fmt)
        self.bank_dn = ft.make_bank(*banks[1], fmt=self.ft_fmt)
        self.sets = []
        for i in range(self.NSETS):
            s = seed + 17 * (i + 1)
            ids = (synth.routes_fast(T, k, E, s, device) if active == k and T * k > 256 else
                   synth.routes(T, k, E, s, active_per_token=active, device=device))
            self.sets.append((synth.activations_bf16(T, H, s, device), ids,
                              synth.routing_weights(T, k, s, device)))
        self.shape = ft.moe_shape(T, H, I, k, E, fmt=self.ft_fmt, path=path)
        # the path the library takes (path 0 is its automatic choice): the route-slot path,
        # or the grouped path with SiLU-and-mul fused into the gate/up GEMM (no fp32 gate/up
        # buffer in the workspace) or in its own kernel
        lay = ft.ftmoe_forward_workspace_layout(self.shape)
        self.decode = lay["partials_bytes"] > 0  # the fused decode kernel (path 4)
        self.grouped = path != 1 and not self.decode
        self.fused = self.grouped and lay["gateup_bytes"] == 0
        # the combine inside the down GEMM (arrival counters in the workspace, no combine launch)
        self.comb = self.grouped and lay["counters_bytes"] > 0
        self.ws = torch.empty(ft.ftmoe_forward_workspace_bytes(self.shape), dtype=torch.uint8, device=device)
        self.x_in = torch.empty(T, H, dtype=torch.bfloat16, device=device)
        self.ids_in = torch.empty(T, k, dtype=torch.int32, device=device)
        self.w_in = torch.empty(T, k, dtype=torch.float32, device=device)
        self.out = torch.empty(T, H, dtype=torch.bfloat16, device=device)
        # kernels per forward: quantize, [segment, gather,] gate/up, SiLU-and-mul, down, combine;
        # FP8 on the grouped path quantizes and segments in one launch, and the fused path has
        # no SiLU-and-mul launch; each NVFP4 quantizer adds an amax pass and the tensor-scale
        # conversion; MXFP8 quantizes inside the gather (no quantizing launch)
        self.launches_per_step = ((5 if path == 1 else 7) - (1 if self.fused else 0) - (1 if self.comb else 0) -
                                  (1 if self.grouped and self.fmt in ("fp8", "mxfp8") else 0) +
                                  (4 if self.fmt == "nvfp4" else 0))
        if self.decode:
            self.launches_per_step = 2  # quantize, then the fused kernel

    # algorithmic bytes/flops of one forward on route set i
    def work(self, i):
        _, ids, _ = self.sets[i]
        ids = ids.cpu().numpy()
        T, H, I, k = self.T, self.H, self.I, self.k
        uniq = len(set(int(e) for e in ids.reshape(-1) if e >= 0))
        ra = int((ids >= 0).sum())
        R = T * k
        f = self.fmt
        row = lambda n: code_bytes(f, n) + scale_bytes(f, n)  # noqa: E731 - one quantized row
        w_gu = weight_bytes(f, 2 * I, H)
        w_dn = weight_bytes(f, H, I)
        if self.decode:
            # token rows in, each distinct expert's weights once, the intermediate and down
            # rows of the active routes written and read back once, the output written
            row = lambda n: code_bytes(f, n) + scale_bytes(f, n)  # noqa: E731
            w_gu = weight_bytes(f, 2 * I, H)
            w_dn = weight_bytes(f, H, I)
            gateup = T * H * 2 + T * row(H) + uniq * w_gu + ra * row(I)
            total = (T * H * 2 + T * row(H) + uniq * (w_gu + w_dn) + 2 * ra * row(I) + 2 * ra * H * 4 +
                     T * k * 8 + T * H * 2)
            return dict(bytes=total, gateup_bytes=total, flops=2 * ra * (2 * I * H + H * I),
                        gateup_flops=2 * ra * (2 * I * H + H * I), uniq=uniq, active=ra)
        out_rows = ra if self.grouped else R     # the route-slot path also writes zero rows
        if self.fused:   # gate/up + SiLU-and-mul: writes the re-quantized rows, no fp32 rows
            gateup = uniq * w_gu + ra * row(H) + ra * row(I)
            silu = 0
        else:
            gateup = uniq * w_gu + (ra if self.grouped else T) * row(H) + out_rows * 2 * I * 4
            silu = out_rows * 2 * I * 4 + out_rows * row(I)
        if self.comb:
            # the combine inside the down GEMM: the fp32 rows need not leave L2 (each is
            # written once and read once, within the same block-pair span of the GEMM)
            down = uniq * w_dn + out_rows * row(I)
            comb = T * k * 8 + T * H * 2
        else:
            down = uniq * w_dn + out_rows * row(I) + out_rows * H * 4
            comb = ra * H * 4 + T * k * 8 + T * H * 2
        total = gateup + silu + down + comb
        if f == "nvfp4":
            total += T * H * 2 + out_rows * 2 * I * 4              # amax passes of the tensor scales
        if f == "mxfp8":
            # segment, then the gather reads each bf16 token row once and writes the quantized
            # rows of the active routes
            total += T * k * 4 * 3 + T * H * 2 + ra * row(H)
        else:
            total += T * H * 2 + T * row(H)                        # quantize
            if self.grouped:
                total += T * k * 4 * 3 + ra * row(H) * 2           # segment + gather
        flops = 2 * ra * (2 * I * H + H * I)
        return dict(bytes=total, gateup_bytes=gateup, flops=flops, gateup_flops=2 * ra * 2 * I * H,
                    uniq=uniq, active=ra)

    def load_set(self, i):
        x, ids, w = self.sets[i]
        self.x_in.copy_(x)
        self.ids_in.copy_(ids)
        self.w_in.copy_(w)

    def forward(self, stream=None):
        self.ft.ftmoe_moe_forward(self.shape, self.x_in, self.ids_in, self.w_in, self.bank_gu, self.bank_dn,
                                  self.out, self.ws, stream=stream)

    def dominant_kernel(self):
        """The gate/up GEMM alone, on the rows the forward left in the workspace; on the fused
        decode path the whole forward (its quantizing launch and the fused kernel)."""
        ft = self.ft
        if self.decode:
            return "decode_fused_kernel (+ its quantizing launch; the whole forward)", self.forward
        lay = ft.ftmoe_forward_workspace_layout(self.shape)
        T, H, k = self.T, self.H, self.k
        gu = self.ws[lay["gateup"]:lay["gateup"] + lay["gateup_bytes"]].view(torch.float32).view(T * k, -1)
        if not self.grouped:
            xq = self.ws[lay["x_q"]:lay["x_q"] + T * H].view(T, H)
            xs = self.ws[lay["x_scales"]:lay["x_scales"] + T * (-(-H // 128)) * 4].view(torch.float32).view(T, -1)
            act, routes = ft.make_act(xq, xs), ft.slot_routes(self.ids_in)
            return "stream_gemm_kernel (gate/up, route slots)", lambda: ft.ftmoe_grouped_gemm_gateup(
                act, routes, self.bank_gu, gu, variant=1)
        R = T * k
        f = self.fmt
        rq = self.ws[lay["rows_q"]:lay["rows_q"] + R * code_bytes(f, H)].view(R, -1)
        rs = self.ws[lay["rows_scales"]:lay["rows_scales"] + R * scale_bytes(f, H)]
        rs = rs.view(torch.float32).view(R, -1) if f == "fp8" else rs.view(R, -1)
        off = self.ws[lay["offsets"]:lay["offsets"] + (self.E + 1) * 4].view(torch.int32)
        tile = ft.ftmoe_pick_tile(R, self.E)
        if f == "fp8":
            # (a CTA pair per unit at token tile 128 where the matrix is whole 256-row block pairs)
            pair = tile == 128 and (2 * self.I) % 256 == 0 and H % 128 == 0
            act = ft.make_act(rq, rs)
            kname = (f"tc_gemm_kernel<{tile}, CTA pair> (gate/up, grouped, tcgen05 cta_group::2)" if pair else
                     f"tc_gemm_kernel<{tile}> (gate/up, grouped, tcgen05)")
        elif f == "mxfp8":
            act = ft.make_act(rq, rs, fmt=ft.FMT_MXFP8)
            kname = f"mxfp8_gemm_kernel<{tile}> (gate/up, grouped, tcgen05 block-scaled)"
        else:
            xg = self.ws[lay["x_gscale"]:lay["x_gscale"] + 4].view(torch.float32)
            act = ft.make_act(rq, rs, xg, fmt=ft.FMT_NVFP4)
            kname = f"nvfp4_gemm_kernel<{tile}> (gate/up, grouped, tcgen05 block-scaled)"
        routes = ft.grouped_routes(off)
        if self.fused:
            aq = self.ws[lay["act_q"]:lay["act_q"] + lay["act_q_bytes"]].view(R, -1)
            asc = self.ws[lay["act_scales"]:lay["act_scales"] + lay["act_scales_bytes"]].view(torch.float32).view(R, -1)
            kname = f"tc_gemm_kernel<{tile}, gate/up pairs> (gate/up + SiLU-and-mul + FP8 requant, tcgen05)"
            return kname, lambda: ft.ftmoe_grouped_gemm_gateup_silu(act, routes, self.bank_gu, aq, asc, tok_tile=tile)
        return kname, lambda: ft.ftmoe_grouped_gemm_gateup(act, routes, self.bank_gu, gu, tok_tile=tile, variant=2)


class L2Flush:
    """Replaces L2's contents between timed steps: a 512 MiB write (larger than the 126 MB
    L2), then a 256 MiB read of another buffer, so that the dirty lines the write leaves are
    written back before the timed region instead of during the next kernel's misses."""
    DESC = "flushed before every timed step (512 MiB write, then a 256 MiB read)"

    def __init__(self, device):
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device=device)
        self.r = torch.zeros(64 << 20, dtype=torch.float32, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def time_in_graph(fn, prep, steps):
    """Device time (ms, summed over `steps` replays) of fn between two event nodes recorded
    inside its own CUDA graph, so the graph's own launch latency is not counted; None
    when this PyTorch cannot record events inside a graph."""
    try:
        e0 = torch.cuda.Event(enable_timing=True, external=True)
        e1 = torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return None
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        e0.record()
        fn()
        e1.record()
    torch.cuda.synchronize()
    total = 0.0
    for i in range(steps):
        prep(i)
        g.replay()
        torch.cuda.synchronize()
        total += e0.elapsed_time(e1)
    return total


def event_floor_us(prep, steps, device):
    """Time between two event nodes around a one-element tensor update in its own graph (the
    same method as the kernels' launch_us): the floor that every launch_us figure includes."""
    tiny = torch.zeros(1, device=device)
    ms = time_in_graph(lambda: tiny.add_(1.0), prep, steps)
    return None if ms is None else round(ms * 1e3 / steps, 3)


def time_events(fn, prep, steps, stream):
    """Sum of per-call CUDA-event durations (ms) over `steps` calls; prep() runs outside."""
    total = 0.0
    evs = []
    for i in range(steps):
        prep(i)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    for e0, e1 in evs:
        total += e0.elapsed_time(e1)
    return total


def run_gpu(args, rank, world, local):
    import block_quantized_moe_gb300 as ft
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = MoeWorkload(args.workload, dev)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)

    def prep(i):
        wl.load_set(i % wl.NSETS)
        flush()

    # eager warm-up, then capture one graph of the whole forward (--eager: direct launches,
    # e.g. for profilers that replay kernels one by one)
    wl.load_set(0)
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        wl.forward(stream=side)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    if args.eager:
        run_step = wl.forward
    else:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            wl.forward()
        torch.cuda.synchronize()
        run_step = graph.replay

    for i in range(args.warmup):
        prep(i)
        run_step()
    torch.cuda.synchronize()

    clocks = ClockSampler(dev)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    t_wall = time.perf_counter()
    ms = time_events(run_step, prep, args.steps, stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    ms_max = max_over_ranks(ms, world, dev)
    us_per_call_rank = ms_max * 1e3 / args.steps
    value = ms_max * 1e3 / (args.steps * world)

    # algorithmic work averaged over the sets the timed steps used
    works = [wl.work(i % wl.NSETS) for i in range(args.steps)]
    bytes_avg = float(np.mean([w["bytes"] for w in works]))
    flops_avg = float(np.mean([w["flops"] for w in works]))
    gu_bytes_avg = float(np.mean([w["gateup_bytes"] for w in works]))
    gu_flops_avg = float(np.mean([w["gateup_flops"] for w in works]))
    hbm_peak, bf16_peak, bf16_sus, peak_src = peaks()
    # dense FP8 = 2x bf16 and dense FP4 = 6x bf16 (nominal ratios 4.5 / 2.25 and 13.5 / 2.25)
    mma_peak = (6.0 if wl.fmt == "nvfp4" else 2.0) * bf16_peak
    mma_name = "fp4" if wl.fmt == "nvfp4" else "fp8"

    # dominant kernel alone (gate/up GEMM), captured in a graph so that host-side launch
    # preparation stays out of the timed region; timed by event nodes inside that graph
    # (L2 flushed before each replay), else by events around the graph's launch
    kname, kern = wl.dominant_kernel()
    for i in range(3):
        prep(i)
        kern()
    torch.cuda.synchronize()
    kms = time_in_graph(kern, prep, args.steps)
    k_timing = "event nodes inside the kernel's graph"
    if kms is None:
        kgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(kgraph):
            kern()
        torch.cuda.synchronize()
        kms = time_events(kgraph.replay, prep, args.steps, stream)
        k_timing = "events around a one-kernel graph (includes the graph's launch latency)"
    k_us = kms * 1e3 / args.steps
    k_gbs = gu_bytes_avg / (k_us * 1e-6) / 1e9
    k_tflops = gu_flops_avg / (k_us * 1e-6) / 1e12

    # end to end through the public API: pinned host inputs -> device, forward, output -> host
    hx = [torch.empty(wl.T, wl.H, dtype=torch.bfloat16, pin_memory=True) for _ in range(wl.NSETS)]
    hids = [torch.empty(wl.T, wl.k, dtype=torch.int32, pin_memory=True) for _ in range(wl.NSETS)]
    hw = [torch.empty(wl.T, wl.k, dtype=torch.float32, pin_memory=True) for _ in range(wl.NSETS)]
    for i, (x, ids, w) in enumerate(wl.sets):
        hx[i].copy_(x)
        hids[i].copy_(ids)
        hw[i].copy_(w)
    hout = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, pin_memory=True)

    def e2e_step(i):
        j = i % wl.NSETS
        wl.x_in.copy_(hx[j], non_blocking=True)
        wl.ids_in.copy_(hids[j], non_blocking=True)
        wl.w_in.copy_(hw[j], non_blocking=True)
        run_step()
        hout.copy_(wl.out, non_blocking=True)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_total = 0.0
    for i in range(args.steps):
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_step(i)
        torch.cuda.synchronize()
        e2e_total += time.perf_counter() - t0
    e2e_us = max_over_ranks(e2e_total, world, dev) * 1e6 / (args.steps * world)
    h2d = wl.T * wl.H * 2 + wl.T * wl.k * 4 * 2
    d2h = wl.T * wl.H * 2

    result = {
        "metric": "MoE FFN us/call",
        "value": round(value, 3),
        "unit": "us/call",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max / args.steps, 5),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": vs_pages(wl.name, value),
        "dtype": {"fp8": "fp8-e4m3 (fp32 accumulate)",
                  "mxfp8": "mxfp8-e4m3 with E8M0 scales per 32 (fp32 accumulate)",
                  "nvfp4": "nvfp4-e2m1 with e4m3 block scales (fp32 accumulate)"}[wl.fmt],
        "data": "synthetic (seeded N(0,1) bf16 activations, N(0,0.02) weights quantized by libftmoe)",
        "config": {"workload": wl.name, "tokens": wl.T, "hidden": wl.H, "inter": wl.I, "experts": wl.E,
                   "topk": wl.k, "active_routes_per_token": wl.active, "route_sets_rotated": wl.NSETS,
                   "forward_path": ("fused decode kernel (one launch after quantization)" if wl.decode else
                                    "route slots (streaming kernel)" if not wl.grouped else
                                    ("grouped, SiLU-and-mul fused into the gate/up GEMM" if wl.fused else
                                     "grouped, separate SiLU-and-mul kernel") +
                                    (", combine inside the down GEMM" if wl.comb else "")),
                   "l2": L2Flush.DESC, "parallelism": f"replicas x{world}",
                   "graph": ("direct launches (--eager)" if args.eager else
                             "one CUDA graph replayed; inputs copied in place between steps")},
        "us_per_call_per_gpu": round(us_per_call_rank, 3),
        "hbm_gbs": round(bytes_avg / (us_per_call_rank * 1e-6) / 1e9, 1),
        "hbm_frac_of_peak": round(bytes_avg / (us_per_call_rank * 1e-6) / 1e9 / hbm_peak, 4),
        f"{mma_name}_tflops": round(flops_avg / (us_per_call_rank * 1e-6) / 1e12, 3),
        f"{mma_name}_frac_of_dense_peak": round(flops_avg / (us_per_call_rank * 1e-6) / 1e12 / mma_peak, 5),
        "algorithmic_bytes_per_call": int(bytes_avg),
        "roofline": {"kernel": kname, "bound": "hbm",
                     "achieved": round(k_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(k_gbs / hbm_peak, 4), "traffic": recorded_traffic(wl.name),
                     "launch_us": round(k_us, 3), "timing": k_timing,
                     "event_floor_us": event_floor_us(prep, args.steps, dev),
                     "algorithmic_bytes_per_launch": int(gu_bytes_avg),
                     f"{mma_name}_tflops": round(k_tflops, 2),
                     f"{mma_name}_frac_of_dense_peak": round(k_tflops / mma_peak, 4),
                     "peak_source": peak_src},
        "e2e": {"value": round(e2e_us, 3), "unit": "us/call", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": wl.launches_per_step * args.steps,
        "clocks": clk,
        "wall_s_timed_region": round(t_wall, 4),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl.name, budget_s=args.cpu_budget)
    return result


def run_gather(args, rank, world, local):
    """The gather-alone workload: one ftmoe_gather_rows_scales per step from a CUDA graph,
    the map of the next set copied in and L2 flushed before every step."""
    import block_quantized_moe_gb300 as ft
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    k, T, topk = GATHER_WORKLOADS[args.workload]
    n_dst, ng, nsets = T * topk, -(-k // 128), 8
    seed = 0xF7E00003
    src = synth.random_bytes(T, k, seed, "gather-src", dev)
    sc = synth.uniform_f32(T, ng, 1e-3, 1.0, seed, "gather-scales", dev)
    maps = [synth.randint_map(n_dst, T, seed + i, "gather-map", dev) for i in range(nsets)]
    map_in = torch.empty(n_dst, dtype=torch.int32, device=dev)
    dst = torch.empty(n_dst, k, dtype=torch.uint8, device=dev)
    dsc = torch.empty(n_dst, ng, dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    def step():
        ft.ftmoe_gather_rows_scales(src, sc, map_in, dst, dsc)

    def prep(i):
        map_in.copy_(maps[i % nsets])
        flush()

    prep(0)
    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    for i in range(args.warmup):
        prep(i)
        graph.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(dev)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    ms = time_events(graph.replay, prep, args.steps, stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms_max = max_over_ranks(ms, world, dev)
    us_rank = ms_max * 1e3 / args.steps
    value = ms_max * 1e3 / (args.steps * world)
    kms = time_in_graph(step, prep, args.steps)
    k_timing = "event nodes inside the kernel's graph"
    if kms is None:
        kms, k_timing = ms, "events around the graph's launch"
    k_us = kms * 1e3 / args.steps
    row = k + 4 * ng
    distinct = [len(set(m.cpu().tolist())) for m in maps]
    bytes_avg = float(np.mean([n_dst * row + d * row + 4 * n_dst for d in
                               (distinct[i % nsets] for i in range(args.steps))]))
    hbm_peak, _, _, peak_src = peaks()
    # end to end: source rows, scales and map from pinned host memory, gathered rows back
    hsrc = torch.empty(T, k, dtype=torch.uint8, pin_memory=True)
    hsc = torch.empty(T, ng, dtype=torch.float32, pin_memory=True)
    hmap = [torch.empty(n_dst, dtype=torch.int32, pin_memory=True) for _ in range(nsets)]
    hsrc.copy_(src)
    hsc.copy_(sc)
    for i in range(nsets):
        hmap[i].copy_(maps[i])
    hdst = torch.empty(n_dst, k, dtype=torch.uint8, pin_memory=True)
    hdsc = torch.empty(n_dst, ng, dtype=torch.float32, pin_memory=True)
    e2e_total = 0.0
    for i in range(args.steps + 3):
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        src.copy_(hsrc, non_blocking=True)
        sc.copy_(hsc, non_blocking=True)
        map_in.copy_(hmap[i % nsets], non_blocking=True)
        graph.replay()
        hdst.copy_(dst, non_blocking=True)
        hdsc.copy_(dsc, non_blocking=True)
        torch.cuda.synchronize()
        if i >= 3:
            e2e_total += time.perf_counter() - t0
    e2e_us = max_over_ranks(e2e_total, world, dev) * 1e6 / (args.steps * world)
    result = {
        "metric": "gather us/call", "value": round(value, 3), "unit": "us/call", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": vs_pages(args.workload, value),
        "dtype": "u8 (FP8 bytes) + fp32 scales",
        "data": "synthetic (seeded random FP8 bytes, U(1e-3, 1) scales, randint maps with duplicates)",
        "config": {"workload": args.workload, "k": k, "tokens": T, "topk": topk, "rows": n_dst,
                   "maps_rotated": nsets, "l2": L2Flush.DESC,
                   "parallelism": f"replicas x{world}", "graph": "one CUDA graph replayed; map copied in between steps"},
        "hbm_gbs": round(bytes_avg / (us_rank * 1e-6) / 1e9, 1),
        "algorithmic_bytes_per_call": int(bytes_avg),
        "roofline": {"kernel": "gather_kernel", "bound": "hbm", "achieved": round(bytes_avg / (k_us * 1e-6) / 1e9, 1),
                     "peak": hbm_peak, "unit": "GB/s", "frac": round(bytes_avg / (k_us * 1e-6) / 1e9 / hbm_peak, 4),
                     "traffic": None, "launch_us": round(k_us, 3), "timing": k_timing,
                     "event_floor_us": event_floor_us(prep, args.steps, dev), "peak_source": peak_src},
        "e2e": {"value": round(e2e_us, 3), "unit": "us/call", "h2d_bytes_per_step": T * k + T * ng * 4 + n_dst * 4,
                "d2h_bytes_per_step": n_dst * row},
        "gpu_launches": args.steps, "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline_gather(args.workload, budget_s=min(args.cpu_budget, 10.0))
    return result


# ------------------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# ------------------------------------------------------------------------------------

def _oracle_problem(name, seed=0xF7E00002, max_tokens=None):
    """Inputs of the oracle's sampled call: x, ids, weights of the first max_tokens tokens,
    the full call's token count, the format and the experts the sample uses."""
    T, H, I, E, k, active, _ = WORKLOADS[name]
    fmt = workload_format(name)
    x = synth.activations_bf16(T, H, seed + 17, "cpu")
    ids = (synth.routes_fast(T, k, E, seed + 17, "cpu") if active == k and T * k > 256 else
           synth.routes(T, k, E, seed + 17, active_per_token=active, device="cpu"))
    w = synth.routing_weights(T, k, seed + 17, "cpu")
    if max_tokens is not None:  # the first tokens of the call
        ids, x, w = ids[:max_tokens], x[:max_tokens], w[:max_tokens]
    used = sorted(set(int(e) for e in ids.reshape(-1).tolist() if e >= 0))
    return x.float().numpy(), ids.numpy(), w.numpy(), T, fmt, used


def _numpy_banks(name, used, seed=0xF7E00002):
    """The numpy oracle's lazily quantized banks, the sample's experts quantized up front
    (the quantized bank is an input; it is built before timing)."""
    from oracle import moe as M
    _, H, I, _, _, _, _ = WORKLOADS[name]
    fmt = workload_format(name)
    bg = M.LazyBank(lambda e: synth.expert_weight_fp32(2 * I, H, seed, e, "gateup", "cpu").numpy(), 2 * I, fmt)
    bd = M.LazyBank(lambda e: synth.expert_weight_fp32(H, I, seed, e, "down", "cpu").numpy(), H, fmt)
    for e in used:
        bg.parts(e)
        bd.parts(e)
    return M, bg, bd


def _oracle_token(M, x, ids, w, bg, bd, fmt, t):
    """The numpy oracle's forward for token t alone. FP8 quantizes per token, so one token of
    the call is exact; the NVFP4 tensor scales span the whole call, so there the token is run
    as a call of its own (the same work per token)."""
    if fmt in ("fp8", "mxfp8"):  # scales per row: one token of the call is exact
        M.moe_forward(x, ids, w, bg, bd, fmt=fmt, tokens_subset=[t])
    else:
        M.moe_forward(x[t:t + 1], ids[t:t + 1], w[t:t + 1], bg, bd, fmt="nvfp4")


def _cpp_oracle_call(x, ids, w, used, fmt, H, I, seed=0xF7E00002):
    """The C++ oracle's inputs for a call of these tokens, with the bank compacted to the
    experts they use (expert ids renumbered; the arithmetic does not depend on the
    numbering). The experts' raw weights are drawn and quantized by the C++ oracle's own
    quantizers on all host threads (ctypes and torch release the GIL), before timing.
    Returns a function running the whole call on `threads` host threads."""
    import concurrent.futures
    from oracle import cpu as C
    C.lib()  # raises if the C++ oracle cannot be built or loaded
    remap = np.full(max(used) + 1 if used else 1, -1, np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    ids_c = np.where(ids >= 0, remap[np.maximum(ids, 0)], -1).astype(np.int32)

    def quantized(job):
        e, tag, n, k = job
        raw = synth.expert_weight_fp32(n, k, seed, e, tag, "cpu").numpy()
        if fmt == "fp8":
            return C.quantize_weight_fp8(raw)
        return C.quantize_mxfp8(raw) if fmt == "mxfp8" else C.quantize_nvfp4(raw)

    jobs = [(e, tag, n, k) for e in used for tag, n, k in (("gateup", 2 * I, H), ("down", H, I))]
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, C.hardware_threads())) as ex:
        parts = list(ex.map(quantized, jobs))

    def stack(which, n, k):
        ps = parts[which::2]
        if fmt == "fp8":
            if not ps:
                return np.zeros((0, n, k), np.uint8), np.zeros((0, -(-n // 128), -(-k // 128)), np.float32)
            return np.stack([p[0] for p in ps]), np.stack([p[1] for p in ps])
        if fmt == "mxfp8":
            if not ps:
                return np.zeros((0, n, k), np.uint8), np.zeros((0, n, -(-k // 32)), np.uint8)
            return np.stack([p[0] for p in ps]), np.stack([p[1] for p in ps])
        if not ps:
            return (np.zeros((0, n, k), np.uint8), np.zeros((0, n, -(-k // 16)), np.uint8),
                    np.zeros(0, np.float32))
        return (np.stack([p[0] for p in ps]), np.stack([p[1] for p in ps]),
                np.array([p[2] for p in ps], np.float32))

    bank_g, bank_d = stack(0, 2 * I, H), stack(1, H, I)
    del parts
    return lambda threads: C.moe_forward(x, ids_c, w, bank_g, bank_d, fmt=fmt, threads=threads)


def cpu_baseline(name, budget_s=20.0, min_s=10.0):
    """Time the oracle on the first (at most 8) tokens of a call, taken as a call of their
    own, in repeated calls until at least min_s (stopping at budget_s); scale the time per
    token to one full call. The C++ oracle runs on every host thread; where it cannot be
    built or loaded, the numpy oracle runs on one thread, token by token. FP8 and MXFP8
    quantize per token, so the sample's rows equal the full call's; NVFP4's tensor scales
    span the sample instead (the same work per token)."""
    T_full = WORKLOADS[name][0]
    x, ids, w, T, fmt, used = _oracle_problem(name, max_tokens=min(T_full, 8))
    n = ids.shape[0]
    try:
        from oracle import cpu as C
        run = _cpp_oracle_call(x, ids, w, used, fmt, *WORKLOADS[name][1:3])
        threads = C.hardware_threads()
    except Exception as exc:  # noqa: BLE001 - the baseline leg only
        run, threads, why = None, 1, str(exc).splitlines()[0] if str(exc) else type(exc).__name__
        M, bg, bd = _numpy_banks(name, used)
    t0 = time.perf_counter()
    done = 0
    while True:
        if run is not None:
            run(threads)
            done += n
        else:
            _oracle_token(M, x, ids, w, bg, bd, fmt, done % n)
            done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (el >= min_s and done % n == 0):
            break
    per_call = el / done * T
    if run is not None:
        sample = (f"{done // n} calls of the first {n} of {T} tokens (C++ oracle, float64, "
                  f"{threads} threads), {el:.1f} s, scaled to the full call")
    else:
        sample = (f"{done} token forwards over the first {n} of {T} tokens of one call (numpy float64, "
                  f"single thread; C++ oracle unavailable: {why}), {el:.1f} s, scaled to the full call")
    res = {"value": round(per_call * 1e6, 1), "unit": "us/call", "cores": threads, "kind": "oracle",
           "sample": sample}
    if run is not None and threads > 1:
        # the same sampled call on one thread, once
        t1 = time.perf_counter()
        run(1)
        el1 = time.perf_counter() - t1
        res["single_thread"] = {"value": round(el1 / n * T * 1e6, 1), "unit": "us/call", "cores": 1,
                                "sample": f"1 call of the first {n} of {T} tokens (C++ oracle, one thread), "
                                          f"{el1:.1f} s, scaled to the full call"}
    return res


def _gather_oracle_problem(name, seed=0xF7E00003):
    from oracle import moe as M
    k, T, topk = GATHER_WORKLOADS[name]
    src = synth.random_bytes(T, k, seed, "gather-src", "cpu").numpy()
    sc = synth.uniform_f32(T, -(-k // 128), 1e-3, 1.0, seed, "gather-scales", "cpu").numpy()
    mp = synth.randint_map(T * topk, T, seed, "gather-map", "cpu").numpy()
    return M, src, sc, mp


def cpu_baseline_gather(name, budget_s=10.0):
    """The oracle's gather (numpy indexing, single thread) on the whole call, repeated
    within the budget."""
    M, src, sc, mp = _gather_oracle_problem(name)
    t0 = time.perf_counter()
    n = 0
    while n < 3 or (time.perf_counter() - t0) < min(budget_s, 1.0):
        M.gather_rows_scales(src, sc, mp)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    el = time.perf_counter() - t0
    return {"value": round(el / n * 1e6, 1), "unit": "us/call", "cores": 1, "kind": "oracle",
            "sample": f"{n} whole calls (numpy, single thread), {el:.2f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    if args.workload in GATHER_WORKLOADS:
        M, src, sc, mp = _gather_oracle_problem(args.workload)
        for _ in range(args.warmup):
            M.gather_rows_scales(src, sc, mp)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            M.gather_rows_scales(src, sc, mp)
        us = (time.perf_counter() - t0) / args.steps * 1e6
        return {"impl": "reference", "metric": "gather us/call", "value": round(us, 1), "unit": "us/call",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 4),
                "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
                "config": {"workload": args.workload},
                "cpu_baseline": {"value": round(us, 1), "unit": "us/call", "cores": 1, "kind": "oracle",
                                 "sample": "whole calls (numpy, single thread)"},
                "e2e": {"value": round(us, 1), "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    T_full = WORKLOADS[args.workload][0]
    x, ids, w, T, fmt, used = _oracle_problem(args.workload, max_tokens=min(T_full, 8))
    ns = ids.shape[0]
    try:
        from oracle import cpu as C
        run = _cpp_oracle_call(x, ids, w, used, fmt, *WORKLOADS[args.workload][1:3])
        threads = C.hardware_threads()
        per_step = ns
        what = f"each step: a call of the first {ns} of {T} tokens (C++ oracle, {threads} threads)"
    except Exception:  # noqa: BLE001 - the reference leg only
        run, threads, per_step = None, 1, 1
        what = f"each step: 1 of {T} tokens of one call (numpy oracle, one thread)"
        M, bg, bd = _numpy_banks(args.workload, used)

    def step(i):
        if run is not None:
            run(threads)
        else:
            _oracle_token(M, x, ids, w, bg, bd, fmt, i % ns)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    el = time.perf_counter() - t0
    us = el / (args.steps * per_step) * T * 1e6
    return {"impl": "reference", "metric": "MoE FFN us/call", "value": round(us, 1), "unit": "us/call",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": args.workload},
            "cpu_baseline": {"value": round(us, 1), "unit": "us/call", "cores": threads, "kind": "oracle",
                             "sample": what + ", scaled to the full call"},
            "e2e": {"value": round(us, 1), "unit": "us/call", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ftmoe", choices=["ftmoe", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS) + sorted(GATHER_WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true", help="launch the forward directly instead of a CUDA graph")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_init()
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    elif args.workload in GATHER_WORKLOADS:
        res = run_gather(args, rank, world, local)
    else:
        res = run_gpu(args, rank, world, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
