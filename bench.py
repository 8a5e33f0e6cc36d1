"""Benchmark of the GB300 verification library.

One step = one spec_verify_chain call over one batch of the batched
128K-vocabulary chain workload (B=64, gamma=7, V=128256, bf16 logits,
per-row temperatures with 8 greedy rows): temperature softmax statistics of
every row, accept tests, first-reject scan, residual / bonus draws (all of
the chain hot path; the tree path is measured in ``other_workloads``).

Metric: verified draft positions per second (B * gamma per step), with the
achieved HBM bandwidth (algorithmic logit bytes / call time) against the
measured copy bandwidth in MEASURED_PEAKS.json.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload c3|c5|c2|c1] [--quick]

Under torchrun (N > 1) every rank verifies its own batch (rows starting at
rank_row0(r) of the same seeded synthetic stream): weak scaling with no
collective on the data path; a barrier brackets the timed region and rank 0
reports the max time over ranks.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_verification_48_gb300 import workloads as W  # noqa: E402

METRIC = "verified draft positions/sec and achieved HBM GB/s vs 8 TB/s (1 GB300)"
# Every call is two launches: sv_stats_kernel, then sv_decide_kernel as its
# programmatic dependent (no memset), whatever the rows' alignment.
KERNEL_NAME = "sv_stats_kernel + sv_decide_kernel (one call)"
LAUNCHES_PER_CALL = 2
UNIT = "positions/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["c3", "c5", "c2", "c1", "c4", "draft", "c3u"],
                    default="c3",
                    help="c4 (token trees: mask, greedy walk, KV compaction), draft (the "
                         "draft-side sampler, 1024 rows x 128256 bf16) and c3u (the C3 shape "
                         "with V = 128257: rows off the 16-byte grid) are accepted in --ncu "
                         "mode only")
    ap.add_argument("--quick", action="store_true", help="skip the other workloads")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU work of the oracle baseline (whole passes over the batch)")
    ap.add_argument("--ncu", action="store_true",
                    help="profiling mode: warm-up + steps calls of the workload, nothing else")
    return ap.parse_args()


def rank_row0(rank: int) -> int:
    """First row of rank `rank`'s batch in the seeded row stream (ranks never
    share rows for batches below 100000 rows)."""
    return rank * 100000


def make_workload(name: str, row0: int = 0):
    if name == "c3":
        return W.make_chain("c3_chain_B64_g7_V128256_bf16", 1003, 64, 7, 128256, "bf16",
                            target="zipf", draft_sigma=(0.3, 2.0),
                            temperature=W._c3_temperature, row0=row0)
    if name == "c5":
        return W.make_chain("c5_chain_B256_g4_V256000_bf16_f32probs", 1005, 256, 4, 256000,
                            "bf16", target="zipf", draft_sigma=(0.7, 0.7), temperature=0.8,
                            draft_probs=True, force_accept_every=16, row0=row0)
    if name == "c2":
        return W.make_chain("c2_chain_B1_g5_V32000_bf16_T1.0", 1002, 1, 5, 32000, "bf16",
                            target="zipf", temperature=1.0, row0=row0)
    if name == "c3u":
        return W.make_chain("c3_unaligned_B64_g7_V128257_bf16", 1003, 64, 7, 128257, "bf16",
                            target="zipf", draft_sigma=(0.3, 2.0),
                            temperature=W._c3_temperature, row0=row0)
    if name == "c1":
        return W.make_chain("c1_chain_B1_g4_V1000_f32", 1001, 1, 4, 1000, "f32",
                            target="normal", target_sigma=2.0, draft_sigma=(0.5, 0.5),
                            temperature=1.0, row0=row0)
    raise ValueError(name)


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _code_only(text: str) -> str:
    """C/C++ source with comments removed and whitespace runs collapsed, so
    that the hash below changes with the code, not with its comments."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_sha() -> str:
    """Hash of the code the timed chain kernels compile from: the bf16
    translation unit, the host launch code and every header it includes."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_48_gb300", "csrc")
    files = sorted(f for f in os.listdir(csrc) if f.endswith((".cuh", ".h")))
    files += ["sv_api.cu", "sv_chain_bf16.cu"]
    for f in files:
        h.update(_code_only(open(os.path.join(csrc, f)).read()).encode())
    h.update(_code_only(open(os.path.join(ROOT, "include", "spec_verify.h")).read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per call from the committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", f"dram_traffic_{workload}.txt")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    sha = re.search(r"kernel_source_sha:\s*(\w+)", txt)
    val = re.search(r"dram_bytes_per_call:\s*([0-9.eE+]+)", txt)
    if not sha or not val or sha.group(1) != kernel_source_sha():
        return None
    return float(val.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


class ChainCall:
    """Raw C-ABI call of spec_verify_chain with fixed device buffers."""

    def __init__(self, sv, case, dev, stream):
        self.case = case
        self.sv = sv
        B, g, V = case.B, case.gamma, case.V
        self.dev_in = [case.target.to(dev), case.draft.to(dev), case.draft_tokens.to(dev),
                       case.temperatures.to(dev), case.uniforms.to(dev)]
        self.out = [torch.empty((B, g + 1), dtype=torch.int32, device=dev),
                    torch.empty((B,), dtype=torch.int32, device=dev),
                    torch.empty((B, g, 4), dtype=torch.float32, device=dev),
                    torch.empty((B,), dtype=torch.int32, device=dev)]
        rows = (g + 1) + (0 if case.draft_is_probs else g)
        dt = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}
        nb = sv.spec_verify_workspace_bytes(B, rows, V, dt[case.target.dtype])
        self.ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
        self.stream = stream
        t, d, x, T, u = self.dev_in
        self.args = (ctypes.c_void_p(t.data_ptr()), dt[t.dtype], ctypes.c_void_p(d.data_ptr()),
                     dt[d.dtype], int(case.draft_is_probs), ctypes.c_void_p(x.data_ptr()),
                     ctypes.c_void_p(T.data_ptr()), ctypes.c_void_p(u.data_ptr()), B, g, V,
                     ctypes.c_void_p(self.out[0].data_ptr()),
                     ctypes.c_void_p(self.out[1].data_ptr()),
                     ctypes.c_void_p(self.out[2].data_ptr()),
                     ctypes.c_void_p(self.out[3].data_ptr()),
                     ctypes.c_void_p(self.ws.data_ptr()), ctypes.c_size_t(nb),
                     ctypes.c_void_p(stream.cuda_stream))
        self.fn = sv.lib().spec_verify_chain

    def __call__(self):
        st = self.fn(*self.args)
        if st != 0:
            raise RuntimeError(self.sv.spec_verify_status_string(st))


def time_calls(call, steps, warmup, stream, per_call_events=True):
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)] if per_call_events else None
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(steps):
            if ev:
                ev[i][0].record(stream)
            call()
            if ev:
                ev[i][1].record(stream)
        t1.record(stream)
    torch.cuda.synchronize()
    total_ms = t0.elapsed_time(t1)
    per = [a.elapsed_time(b) for a, b in ev] if ev else [total_ms / steps]
    return total_ms, float(np.mean(per)), float(np.median(per))


def bench_chain_e2e(sv, case, dev, stream, steps):
    """Host buffers in, host results out: H2D of the step's inputs from pinned
    memory, the C-ABI call, D2H of tokens and counts, host sync, per step."""
    host_in = [t.pin_memory() for t in (case.target, case.draft, case.draft_tokens,
                                         case.temperatures, case.uniforms)]
    call = ChainCall(sv, case, dev, stream)
    host_out = [torch.empty_like(call.out[0], device="cpu").pin_memory(),
                torch.empty_like(call.out[1], device="cpu").pin_memory()]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)

    def step():
        with torch.cuda.stream(stream):
            for d, h in zip(call.dev_in, host_in):
                d.copy_(h, non_blocking=True)
            call()
            host_out[0].copy_(call.out[0], non_blocking=True)
            host_out[1].copy_(call.out[1], non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        step()
    t = time.perf_counter()
    for _ in range(steps):
        step()
    dt = time.perf_counter() - t
    return dt, h2d, d2h


def other_workloads(sv, dev, stream, peak):
    """Secondary measurements: the other chain workloads and the tree."""
    out = {}
    # reading a buffer twice the L2 size evicts the inputs and leaves no
    # dirty lines whose write-back would land inside the timed call
    flush = torch.ones(128 * 1024 * 1024, dtype=torch.float16, device=dev)
    for name, steps in (("c5", 200), ("c2", 2000), ("c1", 2000)):
        case = make_workload(name)
        call = ChainCall(sv, case, dev, stream)
        call()
        torch.cuda.synchronize()
        nacc = call.out[1].cpu().numpy()
        nbytes = W.chain_algorithmic_bytes(case, nacc)
        # flush L2 between calls for the small workloads; time each call alone
        times = []
        for i in range(min(steps, 200)):
            with torch.cuda.stream(stream):
                flush.sum()  # on the timed stream, so it never overlaps the call
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            b.synchronize()
            times.append(a.elapsed_time(b))
        ms = float(np.median(times))
        out[case.name] = {"us_per_call": ms * 1e3, "positions_per_s": case.B * case.gamma / (ms * 1e-3),
                          "GBps": nbytes / (ms * 1e-3) / 1e9, "frac_of_peak": nbytes / (ms * 1e-3) / 1e9 / peak,
                          "algorithmic_bytes": nbytes, "l2": "flushed before each call (256 MB read)"}
        if name in ("c2", "c1"):
            # the same single-round call, 100 times in one CUDA graph: the
            # device time per call without host launch overhead
            label = case.name + "_graph100"
            try:
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph, stream=stream):
                    for _ in range(100):
                        call()
                gt = []
                # a replay runs on the current stream: make that the timed one
                with torch.cuda.stream(stream):
                    graph.replay()
                    torch.cuda.synchronize()
                    for _ in range(20):
                        a = torch.cuda.Event(enable_timing=True)
                        b = torch.cuda.Event(enable_timing=True)
                        a.record(stream)
                        graph.replay()
                        b.record(stream)
                        b.synchronize()
                        gt.append(a.elapsed_time(b) / 100)
                gms = float(np.median(gt))
                out[label] = {"us_per_call": gms * 1e3,
                              "positions_per_s": case.B * case.gamma / (gms * 1e-3),
                              "l2": "inputs L2-resident (100 calls back to back per replay)"}
                del graph
            except Exception as e:  # report, never break the bench line
                out[label] = {"error": repr(e)[:200]}
    # C1 and C2 as batches of independent rounds in one call each (the
    # throughput a batched decode loop sees); C1's batch fits in L2 and is
    # flushed before each call, C2's 1024-round batch (720 MB) is not
    for label, case, steps, flush_each in (
            ("c1_batched_256_rounds", W.c1_chain_fp32_v1000(rounds=256), 200, True),
            ("c2_batched_1024_rounds_T1.0", W.c2_chain_bf16_v32000(1.0, rounds=1024), 50, False)):
        call = ChainCall(sv, case, dev, stream)
        call()
        torch.cuda.synchronize()
        nbytes = W.chain_algorithmic_bytes(case, call.out[1].cpu().numpy())
        if flush_each:
            times = []
            for i in range(steps):
                with torch.cuda.stream(stream):
                    flush.sum()
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                a.record(stream)
                call()
                b.record(stream)
                b.synchronize()
                times.append(a.elapsed_time(b))
            ms = float(np.median(times))
        else:
            total, ms, _ = time_calls(call, steps, 5, stream, per_call_events=False)
        out[label] = {"us_per_call": ms * 1e3, "positions_per_s": case.B * case.gamma / (ms * 1e-3),
                      "GBps": nbytes / (ms * 1e-3) / 1e9,
                      "frac_of_peak": nbytes / (ms * 1e-3) / 1e9 / peak,
                      "algorithmic_bytes": nbytes,
                      "l2": "flushed before each call (256 MB read)" if flush_each
                            else "inputs larger than L2, back-to-back calls"}
        del call
    # rows that do not start on 16-byte boundaries: the C3 shape with
    # V = 128257 (bf16 rows of 256514 bytes)
    try:
        ucase = W.make_chain("c3_unaligned_B64_g7_V128257_bf16", 1003, 64, 7, 128257, "bf16",
                             target="zipf", draft_sigma=(0.3, 2.0),
                             temperature=W._c3_temperature)
        ucall = ChainCall(sv, ucase, dev, stream)
        ucall()
        torch.cuda.synchronize()
        ubytes = W.chain_algorithmic_bytes(ucase, ucall.out[1].cpu().numpy())
        _, ums, _ = time_calls(ucall, 200, 10, stream, per_call_events=False)
        out[ucase.name] = {"us_per_call": ums * 1e3,
                           "positions_per_s": ucase.B * ucase.gamma / (ums * 1e-3),
                           "GBps": ubytes / (ums * 1e-3) / 1e9,
                           "frac_of_peak": ubytes / (ums * 1e-3) / 1e9 / peak,
                           "algorithmic_bytes": ubytes,
                           "rows": "off 16-byte boundaries (masked edge blocks)",
                           "l2": "inputs larger than L2, back-to-back calls"}
        del ucall
    except Exception as e:  # report, never break the bench line
        out["c3_unaligned_B64_g7_V128257_bf16"] = {"error": repr(e)[:200]}
    # draft-side draws (the draft step before verification): 1024 rows of
    # the 128K vocabulary, back to back (262 MB > L2)
    dcase = W.make_draft("draft_sample_B1024_V128256_bf16", 1006, 1024, 128256, "bf16",
                         temperature=lambda b, v: 0.0 if b % 8 == 0 else 0.2 + v)
    dl, dT, du = (t.to(dev) for t in (dcase.logits, dcase.temperatures, dcase.uniforms))
    douts = sv.spec_draft_sample(dl, dT, du, stream=stream)
    dws = torch.zeros(sv.spec_verify_workspace_bytes(dcase.B, 1, dcase.V, 1), dtype=torch.uint8,
                      device=dev)

    def dcall():
        sv.spec_draft_sample(dl, dT, du, out_tokens=douts[0], out_probs=douts[1],
                             out_row_status=douts[2], workspace=dws, stream=stream)
    _, dms, _ = time_calls(dcall, 50, 5, stream, per_call_events=False)
    dbytes = dcase.B * dcase.V * 2 + dcase.B * 8
    out[dcase.name] = {"us_per_call": dms * 1e3, "rows_per_s": dcase.B / (dms * 1e-3),
                       "GBps": dbytes / (dms * 1e-3) / 1e9,
                       "frac_of_peak": dbytes / (dms * 1e-3) / 1e9 / peak,
                       "algorithmic_bytes": dbytes,
                       "l2": "inputs larger than L2, back-to-back calls"}
    del dl, dT, du, douts, dws
    tree = W.c4_tree_f16_v32000()
    args = [t.to(dev) for t in (tree.node_logits, tree.parent, tree.node_tokens)]
    res = sv.spec_verify_tree_greedy(*args, tree.max_depth, stream=stream)
    ws = torch.zeros(sv.spec_verify_workspace_bytes(tree.B, tree.N, tree.V, 2), dtype=torch.uint8,
                     device=dev)
    times = []
    for i in range(200):
        with torch.cuda.stream(stream):
            flush.sum()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        sv.spec_verify_tree_greedy(*args, tree.max_depth, out_path=res[0], out_tokens=res[1],
                                   out_num_accepted=res[2], out_row_status=res[3], workspace=ws,
                                   stream=stream)
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    ms = float(np.median(times))
    nbytes = W.tree_algorithmic_bytes(tree)
    out[tree.name] = {"us_per_call": ms * 1e3, "positions_per_s": tree.B * (tree.N - 1) / (ms * 1e-3),
                      "GBps": nbytes / (ms * 1e-3) / 1e9, "frac_of_peak": nbytes / (ms * 1e-3) / 1e9 / peak,
                      "algorithmic_bytes": nbytes, "l2": "flushed before each call (256 MB read)"}

    def flushed(call, n=200):
        ts = []
        for _ in range(n):
            with torch.cuda.stream(stream):
                flush.sum()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return float(np.median(ts))

    # the tree's attention mask for the same 16 trees of 64 nodes
    mres = sv.spec_tree_mask(args[1], stream=stream)
    ms = flushed(lambda: sv.spec_tree_mask(args[1], out_mask=mres[0], out_depth=mres[1],
                                           out_row_status=mres[2], stream=stream))
    mbytes = tree.B * tree.N * 4 + mres[0].numel() * 8 + mres[1].numel() * 4
    out["tree_mask_B16_N64"] = {"us_per_call": ms * 1e3, "GBps": mbytes / (ms * 1e-3) / 1e9,
                                "algorithmic_bytes": mbytes,
                                "l2": "flushed before each call (256 MB read)"}
    # KV compaction of the walked paths: a [32 layers, 16 trees, 4160 slots]
    # cache of 4 KB slot rows (8 KV heads x 128 x K and V, bf16), context 4096
    L_, S_, row = 32, 4096 + tree.N, 4096
    kvc = torch.empty((L_ * tree.B, S_, row // 2), dtype=torch.bfloat16, device=dev)
    kbase = torch.full((L_ * tree.B,), 4096, dtype=torch.int32, device=dev)
    kpath = res[0].repeat(L_, 1).contiguous()
    knacc = res[2].repeat(L_).contiguous()
    kout = sv.spec_tree_kv_compact(kvc, kbase, kpath, knacc, stream=stream)
    ms = flushed(lambda: sv.spec_tree_kv_compact(kvc, kbase, kpath, knacc, out_length=kout[0],
                                                 out_row_status=kout[1], stream=stream))
    kbytes = int(knacc.sum().item()) * row * 2
    out["kv_compact_L32_B16_S4160_row4KB"] = {
        "us_per_call": ms * 1e3, "GBps": kbytes / (ms * 1e-3) / 1e9,
        "algorithmic_bytes": kbytes, "l2": "flushed before each call (256 MB read)"}
    del kvc, flush
    # multi-round simulation through the draft sampler and the chain verifier:
    # 1024 sequences x 64 tokens, gamma = 4, a p / q pair of overlap 0.8, V = 32000
    from speculative_decoding_verification_48_gb300 import simulate
    with torch.cuda.stream(stream):
        r = simulate.simulate(4, 0.8, sequences=1024, tokens=64, V=32000, c=0.05, seed=1,
                              device=dev)
    out["simulate_g4_alpha0.8_S1024_V32000_f32"] = {
        "tokens_per_round": r.tokens_per_round, "tokens_per_round_se": r.tokens_per_round_se,
        "model_tokens_per_round": r.model_tokens_per_round, "speedup_model_c0.05": r.speedup_model,
        "rounds": r.rounds, "us_per_round": r.us_per_round,
        "note": "us_per_round: device time between events around one draft-sample + verify "
                "pair over all 1024 sequences, host launch gaps included"}
    return out


def host_cpu():
    """The host's logical CPU count and CPU model (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        m = re.search(r"^Model name:\s*(.+)$", out, flags=re.M)
        model = m.group(1).strip() if m else None
    except (OSError, subprocess.SubprocessError):
        pass
    if not model and os.path.exists("/proc/cpuinfo"):
        txt = open("/proc/cpuinfo").read()
        m = re.search(r"^(model name|Hardware|CPU part)\s*:\s*(.+)$", txt, flags=re.M)
        model = m.group(2).strip() if m else None
    return os.cpu_count(), model


def cpu_baseline(case, seconds):
    """The float64 oracle as it stands, single process pinned to one core:
    whole passes over the workload's batch rows, repeated until about
    `seconds` of CPU work."""
    import oracle
    args = case.numpy64()
    aff = os.sched_getaffinity(0) if hasattr(os, "sched_getaffinity") else None
    if aff:
        os.sched_setaffinity(0, {min(aff)})
    try:
        passes, dt = 0, 0.0
        while dt < seconds or passes == 0:
            t = time.perf_counter()
            oracle.verify_chain(*args)
            dt += time.perf_counter() - t
            passes += 1
    finally:
        if aff:
            os.sched_setaffinity(0, aff)
    return passes * case.B * case.gamma / dt, dt, passes


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, dev):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(a, world, rank):
    """The oracle on the host cores, same workload, metric and unit; each step
    verifies one batch row of it (a bounded sample)."""
    if rank != 0:
        return
    case = make_workload(a.workload)
    import oracle
    B = case.B
    budget_s = 120.0
    one = case.select([0]).numpy64()
    t = time.perf_counter()
    oracle.verify_chain(*one)
    row_s = time.perf_counter() - t
    steps = max(3, min(a.steps, int(budget_s / max(row_s, 1e-6))))
    warm = min(a.warmup, 3)
    for i in range(warm):
        oracle.verify_chain(*case.select([i % B]).numpy64())
    args = [case.select([i % B]).numpy64() for i in range(steps)]
    t = time.perf_counter()
    for x in args:
        oracle.verify_chain(*x)
    dt = time.perf_counter() - t
    value = steps * case.gamma / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": a.gpus, "steps": steps, "steps_requested": a.steps, "warmup": warm,
            "ms_per_step": dt / steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": case.name, "global_batch": B, "gamma": case.gamma,
                       "V": case.V, "step_sample": "one batch row per step"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{steps} batch rows of {case.name}, one per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    a = parse()
    world, rank, local = dist_setup(a.gpus)
    if a.impl == "reference":
        run_reference(a, world, rank)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    from speculative_decoding_verification_48_gb300 import build
    build.build()
    import speculative_decoding_verification_48_gb300 as sv
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    peak, peak_kind = measured_peak()

    if a.ncu and a.workload == "c4":
        # the tree path of one decoding step: the ancestor mask of the 16
        # trees of 64 nodes, the greedy walk, then the KV compaction of the
        # walked paths in a [32 layers x 16 trees, 320 slots, 4 KB] cache
        # (context 256: the moved rows are the same as at any context, and
        # the cache stays under 1 GB for full profiler captures)
        tree = W.c4_tree_f16_v32000()
        targs = [t.to(dev) for t in (tree.node_logits, tree.parent, tree.node_tokens)]
        kvc = torch.zeros((32 * tree.B, 256 + tree.N, 2048), dtype=torch.bfloat16, device=dev)
        kbase = torch.full((32 * tree.B,), 256, dtype=torch.int32, device=dev)
        for _ in range(1 + a.warmup + a.steps):
            sv.spec_tree_mask(targs[1], stream=stream)
            path, _, nacc, _ = sv.spec_verify_tree_greedy(*targs, tree.max_depth, stream=stream)
            sv.spec_tree_kv_compact(kvc, kbase, path.repeat(32, 1).contiguous(),
                                    nacc.repeat(32).contiguous(), stream=stream)
        torch.cuda.synchronize()
        return
    if a.ncu and a.workload == "draft":
        # the draft-side sampler: 1024 rows of the 128K vocabulary (262 MB)
        dcase = W.make_draft("draft_sample_B1024_V128256_bf16", 1006, 1024, 128256, "bf16",
                             temperature=lambda b, v: 0.0 if b % 8 == 0 else 0.2 + v)
        dl, dT, du = (t.to(dev) for t in (dcase.logits, dcase.temperatures, dcase.uniforms))
        for _ in range(1 + a.warmup + a.steps):
            sv.spec_draft_sample(dl, dT, du, stream=stream)
        torch.cuda.synchronize()
        return
    case = make_workload(a.workload, row0=rank_row0(rank))
    call = ChainCall(sv, case, dev, stream)
    call()
    torch.cuda.synchronize()
    if a.ncu:
        for _ in range(a.warmup + a.steps):
            call()
        torch.cuda.synchronize()
        return
    nacc = call.out[1].cpu().numpy()
    alg_bytes = W.chain_algorithmic_bytes(case, nacc)
    positions = case.B * case.gamma
    l2_bytes = 129 * 1024 * 1024
    input_bytes = sum(t.numel() * t.element_size() for t in call.dev_in)

    barrier(world)
    with ClockSampler(local) as clk:
        # two events bracket the K back-to-back calls: an event recorded
        # between calls would sit between one call's kernels and the next
        # call's, and break the launch chaining the calls use
        total_ms, mean_call_ms, _ = time_calls(call, a.steps, a.warmup, stream,
                                               per_call_events=False)
    barrier(world)
    total_ms = max_over_ranks(total_ms, world, dev)
    ms_per_step = total_ms / a.steps
    value = world * positions * a.steps / (total_ms * 1e-3)

    e2e_dt, h2d, d2h = bench_chain_e2e(sv, case, dev, stream, a.e2e_steps)
    e2e_dt = max_over_ranks(e2e_dt, world, dev)
    e2e_value = world * positions * a.e2e_steps / e2e_dt

    achieved = alg_bytes / (mean_call_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": case.meta["dtype"],
        "data": "synthetic (seeded; stands in for the pages' XSum/HumanEval/WMT workloads)",
        "config": {"workload": case.name, "global_batch": case.B * world, "gamma": case.gamma,
                   "V": case.V, "seq_len": None, "parallelism": f"independent batch rows x{world}",
                   "l2": (f"inputs larger than L2 ({input_bytes / 1e6:.0f} MB > "
                          f"{l2_bytes / 1e6:.0f} MB)" if input_bytes > l2_bytes else
                          "inputs smaller than L2")},
        "positions_per_step": positions,
        "algorithmic_bytes_per_call": alg_bytes,
        "call_us_mean": mean_call_ms * 1e3,
        "hbm_GBps": achieved, "frac_of_8TBps_nominal": achieved / 8000.0,
        "mean_accepted": float(nacc.mean()),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} (copy bandwidth)",
                     "traffic": ncu_traffic(a.workload),
                     "kernel": KERNEL_NAME},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": a.e2e_steps},
        "gpu_launches": LAUNCHES_PER_CALL * a.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1:
        # the same call with L2 flushed before each call (a 256 MB read on the
        # call's stream), beside the back-to-back figure above
        flush = torch.ones(128 * 1024 * 1024, dtype=torch.float16, device=dev)
        ft = []
        for _ in range(200):
            with torch.cuda.stream(stream):
                flush.sum()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            e1.synchronize()
            ft.append(e0.elapsed_time(e1))
        del flush
        fms = float(np.median(ft))
        line["l2_flushed"] = {"us_per_call": fms * 1e3,
                              "positions_per_s": positions / (fms * 1e-3),
                              "GBps": alg_bytes / (fms * 1e-3) / 1e9,
                              "frac_of_peak": alg_bytes / (fms * 1e-3) / 1e9 / peak,
                              "calls": len(ft),
                              "how": "median of single calls, each after a 256 MB read on "
                                     "the call's stream"}
        v, dt, passes = cpu_baseline(case, a.cpu_seconds)
        nproc, model = host_cpu()
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "host_nproc": nproc, "host_cpu": model,
                                "sample": f"{passes} passes over the {case.B} batch rows of "
                                          f"{case.name} ({dt:.1f} s, single process pinned "
                                          f"to one core)"}
        if not a.quick:
            line["other_workloads"] = other_workloads(sv, dev, stream, peak)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
