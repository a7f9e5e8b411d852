#!/usr/bin/env python3
"""Benchmark: E8 lattice KV-cache compress + decompress on one GB300 per rank.

One step = the whole hot path over the Llama-3.1-8B-shaped cache (32 layers,
batch 4, 8 KV heads, 32768 tokens, head_dim 128, fp16; K2V2, group 64, relaxed
E8 unless --strict): compress K and V (RoPE removal, Hadamard, group scale, E8
nearest point, 2-bit packing), then decompress the buffer back to fp16 K and V.

value = fp16 K+V bytes consumed by compression plus fp16 K+V bytes produced by
decompression, per second of device time (inputs resident in HBM; they are
16 GiB, far larger than L2, so no flush is needed between steps).

Prints one JSON line on rank 0.  `--impl reference` times the CPU oracle (the
stand-in for the method's CPU-bound compression loop) on a bounded sample of
the same workload instead.
"""
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "e8_lattice_vector_gb300", "csrc")


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="llama31_8b")
    ap.add_argument("--strict", action="store_true", help="strict E8 parity instead of relaxed")
    ap.add_argument("--joint", action="store_true", help="strict E8 in the joint 8b-bit format (no coset words)")
    ap.add_argument("--bits", default=None, help="K,V code widths (e.g. 2,2): the config's first mode with them")
    ap.add_argument("--delta-chunk", type=int, default=None,
                    help="temporal delta restart interval instead of the config's (0: none; >= tokens: one chain)")
    ap.add_argument("--e2e-steps", type=int, default=4)
    ap.add_argument("--fused-steps", type=int, default=10, help="timed nq_roundtrip_kv calls (0: skip)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def _peak_hbm():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _code_lines(text):
    """The source's code without // comments, blank lines or indentation: a
    comment edit leaves the kernels, and so the hash, unchanged."""
    out = []
    for line in text.splitlines():
        code = line.split("//", 1)[0].strip()
        if code:
            out.append(code)
    return "\n".join(out)


def _kernel_src_hash(src_dir=None):
    h = hashlib.sha256()
    d = src_dir or CSRC
    for f in sorted(os.listdir(d)):
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            h.update(f.encode() + _code_lines(fh.read()).encode())
    return h.hexdigest()[:16]


def _traffic_record(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[kernel]
        if rec.get("src_hash") == _kernel_src_hash():
            return rec
    except Exception:
        pass
    return None


def _pick_params(cfg, a):
    """The config's first codec mode with the requested parity (and code widths,
    --bits); --joint turns it into the strict joint format, --delta-chunk sets
    the delta restart interval."""
    from e8_lattice_vector_gb300 import CodecParams

    strict = a.strict or a.joint
    modes = list(cfg.modes)
    if getattr(a, "bits", None):
        kb, vb = (int(x) for x in a.bits.split(","))
        modes = [m for m in modes if (m.key_bits, m.value_bits) == (kb, vb)]
        if not modes:
            raise SystemExit("config %s has no K%dV%d mode" % (cfg.name, kb, vb))
    params = ([m for m in modes if bool(m.strict) == strict] or modes)[0]
    delta = params.delta_chunk if getattr(a, "delta_chunk", None) is None else a.delta_chunk
    return CodecParams(params.key_bits, params.value_bits, params.group_size, 2 if a.joint else params.strict, delta,
                       params.rope_theta)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                 "-lms", "50", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            with open(self.path) as f:
                for line in f:
                    p = [x.strip() for x in line.split(",")]
                    if len(p) < 9:
                        continue
                    try:
                        sm.append(float(p[1]))
                        smax.append(float(p[2]))
                    except ValueError:
                        continue
                    for n, v in zip(names, p[5:9]):
                        if v.lower() == "active":
                            reasons.add(n)
            os.unlink(self.path)
        except Exception:
            return None
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ multi-rank


def dist_max(x, device=None):
    """Max of a float over all ranks (the identity on one process)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world, bytes_per_rank, ms):
    """Whole-job rate: every rank processed bytes_per_rank in at most ms."""
    return world * bytes_per_rank / (ms * 1e-3) / 1e9


# ----------------------------------------------------------------- our arm


def _free_port():
    import socket

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_ranks(gpus, argv, script=None):
    """Start `gpus` ranks of `script` (this file by default) under
    torch.distributed.run on this node, one process per GPU, rendezvous on
    127.0.0.1; returns the launcher's exit status.  Used when --gpus N > 1 is
    given without a torchrun environment."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(gpus),
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           script or os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd)


def init_ranks():
    """(world, rank, local rank) from the torchrun environment; joins the
    process group when there is more than one rank (NCCL on GPUs, gloo
    otherwise).  Every rank then works on its own replica of the cache: the
    slices are independent, so nothing is exchanged on the data path."""
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def run_ours(a):
    import torch
    import torch.distributed as dist

    from e8_lattice_vector_gb300 import build as nqbuild

    world, rank, local = init_ranks()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    nqbuild.build()
    import e8_lattice_vector_gb300 as nq
    from e8_lattice_vector_gb300.synth import CONFIGS, make_cache

    cfg = CONFIGS[a.config]
    params = _pick_params(cfg, a)
    K, V = make_cache(cfg, device=dev)
    rope = nq.RopeTable.build(cfg.tokens, cfg.head_dim, params.rope_theta, device=dev)
    lay = nq.plan(cfg.shape, params)
    buf = torch.empty(int(lay.total_bytes), dtype=torch.uint8, device=dev)
    ws = nq.workspace(int(lay.workspace_bytes), dev)  # a temporal delta's decompression scratch
    K2 = torch.empty_like(K)
    V2 = torch.empty_like(V)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        nq.compress_kv(K, V, params, rope, out=buf)
        if ev:
            ev[1].record(stream)
        nq.decompress_kv(buf, cfg.shape, params, rope, K_out=K2, V_out=V2, ws=ws)
        if ev:
            ev[2].record(stream)

    for _ in range(max(a.warmup, 0)):
        step()
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(a.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(a.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    comp_ms = [e[0].elapsed_time(e[1]) for e in evs]
    decomp_ms = [e[1].elapsed_time(e[2]) for e in evs]
    total_ms = dist_max(total_ms, dev)

    # ---- the one-pass round trip (nq_roundtrip_kv) on the same cache, timed
    # the same way after the headline steps: fp16 in, fp16 out, no records
    fused = None
    if a.fused_steps > 0:
        for _ in range(max(a.warmup, 0)):
            nq.roundtrip_kv(K, V, params, rope, K_out=K2, V_out=V2)
        fe = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        torch.cuda.synchronize(dev)
        fe[0].record(stream)
        for _ in range(a.fused_steps):
            nq.roundtrip_kv(K, V, params, rope, K_out=K2, V_out=V2)
        fe[1].record(stream)
        torch.cuda.synchronize(dev)
        fused_ms = dist_max(fe[0].elapsed_time(fe[1]) / a.fused_steps, dev)
        fused = {"ms": round(fused_ms, 4), "gbs": round(whole_job_gbs(world, 2 * cfg.fp16_bytes, fused_ms), 2),
                 "steps": a.fused_steps, "launches": "key + value",
                 "what": "nq_roundtrip_kv: the same reconstruction without the compressed intermediate"}

    # ---- end to end through the public API with pinned host buffers: per layer,
    # upload K, V (copy stream), compress + decompress (compute stream), download
    # the reconstructed K, V (second copy stream); layers overlap across streams
    e2e = None
    if a.e2e_steps > 0:
        hK = torch.empty(K.shape, dtype=K.dtype, pin_memory=True)
        hV = torch.empty(V.shape, dtype=V.dtype, pin_memory=True)
        hK.copy_(K)
        hV.copy_(V)
        oK = torch.empty_like(hK, pin_memory=True)
        oV = torch.empty_like(hV, pin_memory=True)
        nl = cfg.layers
        lshape = (1,) + tuple(cfg.shape[1:])
        llay = nq.plan(lshape, params)
        lbufs = [torch.empty(int(llay.total_bytes), dtype=torch.uint8, device=dev) for _ in range(nl)]
        lws = nq.workspace(int(llay.workspace_bytes), dev)
        s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
        ev_in = [torch.cuda.Event() for _ in range(nl)]
        ev_cmp = [torch.cuda.Event() for _ in range(nl)]

        def e2e_step():
            for l in range(nl):
                with torch.cuda.stream(s_in):
                    K[l].copy_(hK[l], non_blocking=True)
                    V[l].copy_(hV[l], non_blocking=True)
                    ev_in[l].record(s_in)
                with torch.cuda.stream(s_cmp):
                    s_cmp.wait_event(ev_in[l])
                    nq.compress_kv(K[l:l + 1], V[l:l + 1], params, rope, out=lbufs[l])
                    nq.decompress_kv(lbufs[l], lshape, params, rope, K_out=K2[l:l + 1], V_out=V2[l:l + 1], ws=lws)
                    ev_cmp[l].record(s_cmp)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_cmp[l])
                    oK[l].copy_(K2[l], non_blocking=True)
                    oV[l].copy_(V2[l], non_blocking=True)

        def sync_streams():
            for st in (s_in, s_cmp, s_out):
                st.synchronize()

        e2e_step()
        sync_streams()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(s_in)
        for _ in range(a.e2e_steps):
            e2e_step()
        s_out.wait_stream(s_in)
        s_out.wait_stream(s_cmp)
        e1.record(s_out)
        torch.cuda.synchronize(dev)
        e2e_ms = e0.elapsed_time(e1) / a.e2e_steps
        e2e_ms = dist_max(e2e_ms, dev)
        e2e = {"value": round(whole_job_gbs(world, 2 * cfg.fp16_bytes, e2e_ms), 2), "unit": "GB/s",
               "h2d_bytes_per_step": int(hK.numel() * 2 + hV.numel() * 2),
               "d2h_bytes_per_step": int(oK.numel() * 2 + oV.numel() * 2),
               "ms_per_step": round(e2e_ms, 3),
               "pipeline": "per layer on three streams: upload, compress+decompress, download"}
        del hK, hV, oK, oV, lbufs

    # ---- algorithmic bytes and roofline
    rows = cfg.rows
    fp16_row = cfg.head_dim * 2
    cos_row = 0 if int(params.strict) == 2 else 2  # the joint format has no coset words
    rec_row = {"k": lay.k_idx_row_bytes + cos_row + lay.scales_per_row * 2,
               "v": lay.v_idx_row_bytes + cos_row + lay.scales_per_row * 2}
    alg_bytes = rows * (2 * fp16_row + rec_row["k"] + rec_row["v"])  # one direction, K + V
    comp_avg = sum(comp_ms) / len(comp_ms)
    decomp_avg = sum(decomp_ms) / len(decomp_ms)
    peak, peak_kind = _peak_hbm()
    # one "launch" of the compress (decompress) kernel = one nq_compress_kv (nq_decompress_kv)
    # call: its key launch and its value launch, timed together with CUDA events
    kernels = {
        "compress": {"ms": round(comp_avg, 4), "gbs": round(alg_bytes / (comp_avg * 1e-3) / 1e9, 1),
                     "launches": "key + value"},
        "decompress": {"ms": round(decomp_avg, 4), "gbs": round(alg_bytes / (decomp_avg * 1e-3) / 1e9, 1),
                       "launches": "key + value"},
    }
    for kname in kernels:
        kernels[kname]["frac_of_peak"] = round(kernels[kname]["gbs"] / peak, 4)
    dom = "compress" if comp_avg >= decomp_avg else "decompress"
    achieved = kernels[dom]["gbs"]
    trec = _traffic_record(dom) if a.config == "llama31_8b" else None
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": peak_kind,
                "frac_of_nominal_8000": round(achieved / 8000.0, 4),
                "traffic": (int(trec["dram_bytes_per_call"]) if trec else None),
                "algorithmic_bytes": int(alg_bytes)}

    ms_per_step = total_ms / a.steps
    value = whole_job_gbs(world, 2 * cfg.fp16_bytes, ms_per_step)
    out = {
        "metric": "KV compress/decompress GB/s (fp16 in) on 1 GB300; % of HBM roofline",
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": a.steps,
        "warmup": a.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp16",
        "data": "synthetic",
        "config": {
            "workload": "%s KV cache %s fp16, K%dV%d group %d %s E8, delta %s, compress+decompress round trip"
                        % (cfg.name, list(cfg.shape), params.key_bits, params.value_bits, params.group_size,
                           {0: "relaxed", 1: "strict", 2: "strict (joint format)"}[int(params.strict)], params.delta_chunk or "off"),
            "fp16_bytes_per_direction": cfg.fp16_bytes,
            "l2": "inputs (%.1f GiB) larger than L2; no flush" % (cfg.fp16_bytes / 2 ** 30),
            "parallelism": "replicas" if world > 1 else "single",
        },
        "compress_gbs_fp16": round(cfg.fp16_bytes / (comp_avg * 1e-3) / 1e9, 2),
        "decompress_gbs_fp16": round(cfg.fp16_bytes / (decomp_avg * 1e-3) / 1e9, 2),
        "kernels": kernels,
        "roofline": roofline,
        "clocks": clk,
        "e2e": e2e,
        "fused_round_trip": fused,
        "gpu_launches": 4 * a.steps,
    }
    kv0 = (K[0, 0].cpu(), V[0, 0].cpu()) if rank == 0 and not a.no_cpu_baseline else None
    del K, V, K2, V2, buf, ws
    torch.cuda.empty_cache()
    if kv0 is not None:
        out["cpu_baseline"] = cpu_baseline(cfg, params, a.cpu_seconds, kv0)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


# --------------------------------------------------------- CPU oracle arm


def _oracle_sample(cfg, params, target_s, kv0=None):
    """A bounded sample of the workload: whole (layer 0, batch 0, head) slices of
    K and V (given, or generated on the CPU); returns (round trip callable,
    slices per call, seconds per slice)."""
    import numpy as np
    import torch

    import oracle
    from e8_lattice_vector_gb300.synth import layer_kv

    T, D = cfg.tokens, cfg.head_dim
    if kv0 is None:
        k, v = layer_kv(cfg, 0, device="cpu", batch=1)
        kv0 = (k[0], v[0])
    kb = kv0[0].contiguous().view(torch.int16).numpy().view(np.uint16)  # [H, T, D]
    vb = kv0[1].contiguous().view(torch.int16).numpy().view(np.uint16)
    cs = oracle.rope_table(T, D, params.rope_theta) if params.rope_theta > 0 else None

    def round_trip(nslices):
        for s in range(nslices):
            h = s % kb.shape[0]
            ki = oracle.compress_tensor(kb[h], T, D, params.key_bits, params.group_size, int(params.strict),
                                        params.delta_chunk, cs)
            vi = oracle.compress_tensor(vb[h], T, D, params.value_bits, params.group_size, int(params.strict),
                                        params.delta_chunk, None)
            joint = int(params.strict) == 2
            oracle.decompress_tensor(*ki, 1, T, D, params.key_bits, params.group_size, params.delta_chunk, cs,
                                     joint=joint)
            oracle.decompress_tensor(*vi, 1, T, D, params.value_bits, params.group_size, params.delta_chunk, None,
                                     joint=joint)

    t0 = time.perf_counter()
    round_trip(1)
    per_slice = time.perf_counter() - t0
    n = max(1, int(target_s / max(per_slice, 1e-6)))
    return round_trip, n, per_slice


def _oracle_worker(job):
    """One host core's share of the oracle sample (runs in a spawned process)."""
    import numpy as np  # noqa: F401

    import oracle

    kb, vb, T, D, p, nrep, cs = job
    if kb is None:  # start-up: load the oracle library
        oracle.lib()
        return 0.0
    kb_, vb_, g, strict, delta = p["key_bits"], p["value_bits"], p["group_size"], p["strict"], p["delta_chunk"]
    t0 = time.perf_counter()
    for _ in range(nrep):
        ki = oracle.compress_tensor(kb, T, D, kb_, g, strict, delta, cs)
        vi = oracle.compress_tensor(vb, T, D, vb_, g, strict, delta, None)
        oracle.decompress_tensor(*ki, 1, T, D, kb_, g, delta, cs, joint=strict == 2)
        oracle.decompress_tensor(*vi, 1, T, D, vb_, g, delta, None, joint=strict == 2)
    return time.perf_counter() - t0


class _OraclePool:
    """One spawned process per host core (spawned, never forked: the parent
    holds a CUDA context), each with the oracle loaded."""

    def __init__(self):
        import multiprocessing as mp

        self.cores = max(1, os.cpu_count() or 1)
        self.pool = mp.get_context("spawn").Pool(self.cores)
        self.pool.map(_oracle_worker, [(None, None, 0, 0, None, 0, None)] * self.cores, chunksize=1)

    def close(self):
        self.pool.close()
        self.pool.join()


def _oracle_all_cores(cfg, params, cpu_seconds, kv0, per_slice, op, min_rep=3):
    """The oracle on every host core: each process repeats the round trip of one
    (layer 0, batch 0, head) slice; the wall time of the parallel part is
    timed.  Returns (GB/s, cores, slices, s)."""
    import numpy as np
    import torch

    import oracle

    T, D = cfg.tokens, cfg.head_dim
    kb = kv0[0].contiguous().view(torch.int16).numpy().view(np.uint16)
    vb = kv0[1].contiguous().view(torch.int16).numpy().view(np.uint16)
    cs = oracle.rope_table(T, D, params.rope_theta) if params.rope_theta > 0 else None
    # at least three slices per process: the parallel wall time is then long enough to time stably
    nrep = max(min_rep, int(cpu_seconds / op.cores / max(per_slice, 1e-6)))
    p = {"key_bits": params.key_bits, "value_bits": params.value_bits, "group_size": params.group_size,
         "strict": int(params.strict), "delta_chunk": params.delta_chunk}
    jobs = [(kb[w % kb.shape[0]], vb[w % vb.shape[0]], T, D, p, nrep, cs) for w in range(op.cores)]
    t0 = time.perf_counter()
    op.pool.map(_oracle_worker, jobs, chunksize=1)
    dt = time.perf_counter() - t0
    slices = op.cores * nrep
    fp16 = 2 * 2 * slices * T * D * 2
    return fp16 / dt / 1e9, op.cores, slices, dt


def cpu_baseline(cfg, params, target_s, kv0=None):
    rt, n, per_slice = _oracle_sample(cfg, params, target_s / 2, kv0)
    t0 = time.perf_counter()
    rt(n)
    dt = time.perf_counter() - t0
    fp16 = 2 * 2 * n * cfg.tokens * cfg.head_dim * 2  # K+V, compressed and decompressed
    single = fp16 / dt / 1e9
    if kv0 is None:
        from e8_lattice_vector_gb300.synth import layer_kv

        k, v = layer_kv(cfg, 0, device="cpu", batch=1)
        kv0 = (k[0], v[0])
    op = _OraclePool()
    try:
        _oracle_all_cores(cfg, params, 0.0, kv0, per_slice, op, min_rep=1)  # untimed: warm every process
        gbs, cores, slices, wall = _oracle_all_cores(cfg, params, target_s / 2, kv0, per_slice, op)
    finally:
        op.close()
    return {"value": round(gbs, 5), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "single_core_value": round(single, 5),
            "sample": "(layer 0, batch 0, head) slices of %d tokens, K and V, compress+decompress, plain C: "
                      "%d slices on %d cores in %.1f s (one process per core); %d slices on one core in %.1f s"
                      % (cfg.tokens, slices, cores, wall, n, dt)}


def run_reference(a):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from e8_lattice_vector_gb300.synth import CONFIGS

    cfg = CONFIGS[a.config]
    params = _pick_params(cfg, a)
    from e8_lattice_vector_gb300.synth import layer_kv

    k, v = layer_kv(cfg, 0, device="cpu", batch=1)
    kv0 = (k[0], v[0])
    _, _, per_slice = _oracle_sample(cfg, params, 1.0, kv0)
    per_step_s = max(1.0, a.cpu_seconds / max(a.steps, 1))
    op = _OraclePool()
    try:
        for _ in range(max(a.warmup, 0)):
            _oracle_all_cores(cfg, params, 0.0, kv0, per_slice, op)
        total_bytes, total_s, cores, slices = 0.0, 0.0, 1, 0
        for _ in range(a.steps):
            gbs, cores, n, wall = _oracle_all_cores(cfg, params, per_step_s, kv0, per_slice, op)
            total_bytes += gbs * wall
            total_s += wall
            slices += n
    finally:
        op.close()
    value = total_bytes / total_s
    dt = total_s
    sample = ("%d slices of %d tokens over %d steps (layer 0, batch 0), K and V, compress+decompress, "
              "plain C, one process per core on %d cores" % (slices, cfg.tokens, a.steps, cores))
    out = {
        "impl": "reference",
        "metric": "KV compress/decompress GB/s (fp16 in) on 1 GB300; % of HBM roofline",
        "value": round(value, 5), "unit": "GB/s", "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": round(dt / a.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp16", "data": "synthetic",
        "config": {"workload": "%s KV cache (sampled), K%dV%d group %d %s E8" % (
            cfg.name, params.key_bits, params.value_bits, params.group_size,
            {0: "relaxed", 1: "strict", 2: "strict (joint format)"}[int(params.strict)])},
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main():
    a = _args()
    if a.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_ranks(a.gpus, sys.argv[1:]))
    if a.impl == "reference":
        run_reference(a)
    else:
        run_ours(a)


if __name__ == "__main__":
    main()
