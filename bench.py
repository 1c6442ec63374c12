"""Benchmark of one indexer step on synthetic data.

Headline workload: paged FP8 decode (B=64 sequences, next_n=1, context
lengths U[4096, 32768], 64-token pages in a 40,000-page pool, top-2048
mapped to ragged cache slots).  A step is the whole hot path: paged logits,
per-row top-k, and the top-k -> slot map.

Metric: indexer keys scored per second (the (row, key) pairs that receive a
score per step, over the step time), whole job over all ranks.  Every rank
runs its own independent batch (weak scaling; the path has no exchange
step).  After the headline, the same process measures every other workload
(``per_config``: the contiguous prefill and small cases, the MTP candidate
pipeline, MXFP4 decode, the candidate source, the K/Q producers), each with
its own clock record and rooflines.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..7]
                  [--impl ours|reference] [--no-per-config] [--no-cpu]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "indexer Gkeys scored/s (paged FP8 decode) + top-k rows/s; % of HBM/TC roofline"
UNIT = "Gkeys/s"
WORKLOAD_NAMES = {
    1: "non-paged FP8 logits+top-256, M=16 N=1024 H=64 D=128",
    2: "prefill chunk FP8 logits+top-2048, 2048 rows x 8192 keys, H=64 D=128",
    3: "paged FP8 decode, B=64 next_n=1 ctx U[4096,32768], page 64, top-2048 + slots",
    4: "paged FP8 MTP decode, B=128 next_n=2 lognormal ctx (median 16384), 64 candidate blocks "
       "of 128 per row, top-2048 + ragged slots",
    5: "paged MXFP4 decode, B=32 ctx 131072, page 64, top-2048 + slots",
    6: "candidate source at the config-4 shapes: paged FP8 MTP decode, B=128 next_n=2, every "
       "live key scored with block maxima of 128 keys, top-2048 + ragged slots, the 64 best "
       "blocks per row as the candidate pool",
    7: "K/Q producers of a prefill chunk: 8192 tokens, H=64 D=128 rope_dim=64, MXFP4 keys "
       "(RMS norm, RoPE, quantise) stored into 64-token pages, MXFP4 query heads + weights",
}
PROD_METRIC = "producer Mtokens/s (K norm+RoPE+quantise+store, Q RoPE+quantise); % of HBM roofline"
PROD_UNIT = "Mtok/s"


def _is_producer(case) -> bool:
    from sparse_attention_indexer_mxfp4_gb300.synth import ProducerCase
    return isinstance(case, ProducerCase)


def _metric_unit_div(case):
    """(metric, unit, divisor of work per second) of a workload."""
    if _is_producer(case):
        return PROD_METRIC, PROD_UNIT, 1e6
    return METRIC, UNIT, 1e9


def _work(case) -> int:
    """Units of work of one step: keys scored, or tokens produced."""
    return case.T if _is_producer(case) else case.keys_scored


def producer_bytes(case) -> float:
    """Algorithmic bytes of one producer step: each key read once (bf16) and
    written once (codes + scales), its slot, position and rotary row read
    once; each query head read once (bf16) and written once (codes + scales),
    its weight read and written once; the norm weight once."""
    D, H, T = case.D, case.H, case.T
    out = (D + 4) if case.fmt == 0 else (D // 2 + D // 32)
    per_token = 2 * D + out + 8 + 4 + case.rope_dim * 4
    per_head = 2 * D + (D if case.fmt == 0 else D // 2 + 4) + 8
    return float(T * per_token + T * H * per_head + 4 * D)


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one logits
# stage (the plan kernel and the logits kernel under a candidate plan; the
# block-maxima fill and the logits kernel for the candidate source) from an
# ncu capture, per workload, with a digest of the kernels' sources at capture
# time.  A different digest means the kernel changed
# since and the traffic is reported as null.
LOGITS_SOURCES = ["idx_logits_kernel.cuh", "idx_logits.cuh", "idx_common.cuh", "idx_api.cu"]
NCU_TRAFFIC = {
    2: {"bytes": 18609152 + 7529216, "digest": "0eb22f7a66d754d4",
        "profile": "profiles/logits_traffic_all_configs.md"},
    3: {"bytes": 157697280 + 4507904, "digest": "0eb22f7a66d754d4",
        "profile": "profiles/logits_traffic_all_configs.md"},
    4: {"bytes": 87808 + 189602304 + 5477888, "digest": "0eb22f7a66d754d4",
        "profile": "profiles/logits_traffic_all_configs.md"},
    5: {"bytes": 285833984 + 14241024, "digest": "0eb22f7a66d754d4",
        "profile": "profiles/logits_traffic_all_configs.md"},
    6: {"bytes": 4096 + 413308416 + 18571776, "digest": "0eb22f7a66d754d4",
        "profile": "profiles/logits_traffic_all_configs.md"},
}


def logits_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_attention_indexer_mxfp4_gb300", "csrc")
    for name in LOGITS_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def logits_traffic(config: int):
    rec = NCU_TRAFFIC.get(config)
    if rec is None or rec["digest"] != logits_digest():
        return None
    return rec["bytes"]


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class Clocks:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sms.append(float(parts[1]))
                    maxes.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sms) if sms else None,
                "sm_max_mhz": max(maxes) if maxes else None,
                "reasons": sorted(reasons), "samples": len(sms)}


def _case(cfg: int, shard: int = 0):
    """The workload of one rank: rank r runs shard r (its own values, the
    same shapes and lengths), so per-rank work is fixed as ranks are added."""
    from sparse_attention_indexer_mxfp4_gb300 import synth
    return synth.CONFIGS[cfg](shard)


def max_over_ranks(values, device, world: int):
    """Element-wise maximum of per-rank floats over all ranks (the slowest
    rank sets the job time); a no-op on one rank."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), device=device, dtype=torch.float64)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_value(world: int, keys_per_rank: int, ms_per_step: float, div: float = 1e9) -> float:
    """Whole-job work per second (Gkeys/s by default): every rank does
    keys_per_rank units per step and the step takes the slowest rank's time."""
    return world * keys_per_rank / (ms_per_step * 1e-3) / div


def candidate_tile_logits(case, tile=128) -> int:
    """(row, key) logits the candidates-only logits call writes: every key of
    each row below its end inside the tiles (of `tile` keys) that hold a
    candidate key of some row of the sequence."""
    ke = np.clip(case.row_ends(), 0, case.width).reshape(case.B, case.next_n)
    ks = (np.zeros_like(ke) if case.row_ks is None else
          np.minimum(case.row_ks.reshape(case.B, case.next_n), ke))
    total = 0
    for b in range(case.B):
        hi = int(ke[b].max())
        tiles = np.zeros(-(-hi // tile) + 1, dtype=bool)
        for j in range(case.next_n):
            ids = case.cand[b * case.next_n + j]
            ids = ids[ids >= 0].astype(np.int64)
            lo = int(ks[b, j]) + ids * case.cand_block
            hi_r = np.minimum(lo + case.cand_block, int(ke[b, j]))
            for t0, t1 in zip(lo[lo < hi_r], hi_r[lo < hi_r]):
                tiles[t0 // tile:(t1 - 1) // tile + 1] = True
        idx = np.nonzero(tiles)[0]
        for j in range(case.next_n):
            total += int(np.clip(int(ke[b, j]) - idx * tile, 0, tile).sum())
    return total


def candidate_box_keys(case) -> int:
    """Keys in the 64-key boxes that hold a candidate key of some row of their
    sequence (candidate blocks clipped to each row's [ks, ke))."""
    ke = np.clip(case.row_ends(), 0, case.width).reshape(case.B, case.next_n)
    ks = (np.zeros_like(ke) if case.row_ks is None else
          np.minimum(case.row_ks.reshape(case.B, case.next_n), ke))
    total = 0
    for b in range(case.B):
        hi = int(ke[b].max())
        boxes = np.zeros(-(-hi // 64) + 1, dtype=bool)
        for j in range(case.next_n):
            r = b * case.next_n + j
            ids = case.cand[r]
            ids = ids[ids >= 0].astype(np.int64)
            lo = int(ks[b, j]) + ids * case.cand_block
            hi_r = np.minimum(lo + case.cand_block, int(ke[b, j]))
            for t0, t1 in zip(lo[lo < hi_r], hi_r[lo < hi_r]):
                boxes[t0 // 64:(t1 - 1) // 64 + 1] = True
        idx = np.nonzero(boxes)[0]
        total += int(np.minimum(64, hi - idx * 64).clip(min=0).sum())
    return total


def logits_bytes(case, cand_only: bool = True) -> float:
    """Algorithmic bytes of one logits stage: every live key's values and
    scale read once per sequence (with a candidate mask, only the keys of
    boxes that hold a candidate), the group's queries, weights and candidate
    ids read once, one fp32 logit written per scored (row, key), block-table
    entries read once per page."""
    from sparse_attention_indexer_mxfp4_gb300.synth import FMT_FP8, PagedCase
    D, H = case.D, case.H
    per_key = (D + 4) if case.fmt == FMT_FP8 else (D // 2 + D // 32)
    per_q = H * ((D if case.fmt == FMT_FP8 else D // 2 + D // 32) + 4)
    if isinstance(case, PagedCase):
        ke = np.clip(case.row_ends(), 0, case.width)
        seq_keys = ke.reshape(case.B, case.next_n).max(axis=1)
        if case.cand is not None:
            # gather path: only 64-key boxes holding a candidate key of any
            # row of the sequence are read
            b = float(candidate_box_keys(case)) * per_key
        else:
            b = float(seq_keys.sum()) * per_key
        b += case.rows * per_q
        if case.cand is not None and cand_only:
            b += float(candidate_tile_logits(case)) * 4  # only candidate tiles are written
        else:
            b += float(ke.sum()) * 4
        if getattr(case, "source_block", 0):
            # block maxima: the -inf fill and the atomic raises, one word each
            b += 2.0 * case.rows * -(-case.width // case.source_block) * 4
        b += float(np.ceil(seq_keys / case.page_size).sum()) * 4
        if case.cand is not None:
            b += case.cand.size * 4
        return b
    # contiguous: K read once per row group (it stays in L2), Q once, every
    # column of [0, N) of every row written
    b = case.N * per_key + case.M * per_q + case.M * case.N * 4.0
    return b


def logits_flops(case) -> float:
    return 2.0 * case.H * case.D * case.keys_scored


def candidate_keys(case) -> int:
    """(row, key) pairs inside a row's candidate blocks (clipped to its
    [ks, ke)): the keys a candidate pipeline gives a real score."""
    ke = np.clip(case.row_ends(), 0, case.width).astype(np.int64)
    ks = (np.zeros_like(ke) if case.row_ks is None else
          np.minimum(case.row_ks.astype(np.int64), ke))
    total = 0
    for r in range(case.rows):
        ids = np.unique(case.cand[r][case.cand[r] >= 0].astype(np.int64))
        lo = ks[r] + ids * case.cand_block
        hi = np.minimum(lo + case.cand_block, ke[r])
        total += int(np.maximum(hi - lo, 0).sum())
    return total


def scored_keys(case) -> int:
    """(row, key) pairs a step scores: every live key, or with a candidate
    list only the candidate keys (the dense-equivalent count is
    case.keys_scored)."""
    from sparse_attention_indexer_mxfp4_gb300.synth import PagedCase
    if isinstance(case, PagedCase) and case.cand is not None:
        return candidate_keys(case)
    return case.keys_scored


def topk_bytes(case, with_slots: bool = False) -> float:
    """Algorithmic bytes of one top-k stage: every logit the selection
    ranks read once (the live keys of each row, or only its candidate keys)
    and k int32 indices written per row; the candidate source also reads its
    block maxima and writes its pool.  with_slots (the stage also runs the
    slot map, one idx_topk_ragged_slots call): k int32 slots, a row length
    and an indptr entry written per row."""
    from sparse_attention_indexer_mxfp4_gb300.synth import PagedCase
    if isinstance(case, PagedCase):
        b = 4.0 * scored_keys(case) + 4.0 * case.rows * case.topk
        if case.cand is not None:
            b += 4.0 * case.cand.size
        if getattr(case, "source_block", 0):
            nb = -(-case.width // case.source_block)
            b += 4.0 * case.rows * (nb + case.source_cands)
        if with_slots:
            b += 4.0 * case.rows * (case.topk + 2) + 4.0
        return b
    return 4.0 * float(np.maximum(case.ke - case.ks, 0).sum()) + 4.0 * case.M * case.topk


def measure(cfg: int, args, dev, world: int, rank: int, headline: bool) -> dict:
    """One workload: build it, warm up, time args.steps steps (a CUDA graph
    replay), and return its figures.  Paged workloads rotate over three
    device copies of the K pool, so the pages a step reads were last read two
    steps earlier (the 129 MB L2 holds none of them); the contiguous ones and
    the producers rewrite a 256 MB buffer between steps."""
    import torch
    from sparse_attention_indexer_mxfp4_gb300 import (IndexerStep, ProducerStep,
                                                      idx_get_device_status)
    from sparse_attention_indexer_mxfp4_gb300.synth import PagedCase

    case = _case(cfg, shard=rank)
    prod = _is_producer(case)
    step = (ProducerStep(case, device=dev) if prod else
            IndexerStep(case, device=dev, fused_topk=args.fused_topk,
                        fused_slots=not args.split_slots))
    fused = getattr(step, "fused_topk", False)
    paged = isinstance(case, PagedCase)
    steps = [step] + ([step.twin(kv_copy=True), step.twin(kv_copy=True)] if paged else [])
    metric, unit, div = _metric_unit_div(case)

    for _ in range(args.warmup):  # (the first call also builds and loads the library)
        for st in steps:
            st.run()
    torch.cuda.synchronize()
    assert idx_get_device_status() == 0, f"device status set during warm-up (config {cfg})"
    flush = None
    if not paged:
        flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    clocks = Clocks(dev.index if dev.index is not None else 0)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    timing = time_steps_graph(steps, args.steps, flush, clock_soak_s=0.4)
    if timing is None:
        timing = time_steps_eager(steps, args.steps, flush)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    ms_per_step, logit_ms, topk_ms, loop_ms, mode = timing
    assert idx_get_device_status() == 0, f"device status set during the timed steps (config {cfg})"
    logit_step = sum(logit_ms) / len(logit_ms)
    topk_step = sum(topk_ms) / len(topk_ms)
    ms_per_step, logit_step, topk_step, logit_avg, topk_avg = max_over_ranks(
        [ms_per_step, logit_step, topk_step, loop_ms.get("logits_stage", logit_step),
         loop_ms.get("topk_stage", topk_step)], dev, world)

    keys = _work(case) if prod else scored_keys(case)
    rows = case.rows if paged or prod else case.M
    hbm, bf16, src = _peaks()
    if prod:  # the producers' stage times are the K call and the Q call
        lb = producer_bytes(case)
        ach = lb / (ms_per_step * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(ach / hbm, 4), "traffic": None, "peak_source": f"{src} hbm_gbs",
                "kernel": "producer step: k_store_kernel + q_quant_kernel",
                "algorithmic_bytes_per_launch": lb, "avg_launch_ms": round(ms_per_step, 5)}
    elif not paged and cfg == 2:
        fp8_peak = 2.0 * bf16  # dense fp8 rate = 2x bf16 on this part
        ach = logits_flops(case) / (logit_avg * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(ach, 1), "peak": fp8_peak,
                "unit": "TFLOP/s", "frac": round(ach / fp8_peak, 4),
                "traffic": logits_traffic(cfg),
                "peak_source": f"{src} bf16_tflops x 2 (fp8 dense)", "kernel": "logits_kernel",
                "algorithmic_flops_per_launch": logits_flops(case),
                "avg_launch_ms": round(logit_avg, 5), "stage_ms_in_step": round(logit_step, 5)}
    else:
        lb = logits_bytes(case, cand_only=getattr(step, "cand_topk", False))
        if fused:  # the stage also holds the top-k: one more read of the live logits
            lb += 4.0 * float(np.clip(case.row_ends(), 0, case.width).sum())
        ach = lb / (logit_avg * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(ach / hbm, 4),
                "traffic": None if fused else logits_traffic(cfg),
                "peak_source": f"{src} hbm_gbs",
                "kernel": ("fused logits + top-k stage: top-k plan_kernel, logits_kernel with "
                           "digit-1 histograms, top-k phases_kernel from the filter" if fused
                           else "logits stage: cand_plan_kernel (candidate plan) + "
                           "logits_kernel" if getattr(case, "cand", None) is not None
                           else "logits stage: bmax_fill_kernel + logits_kernel with block "
                           "maxima" if getattr(case, "source_block", 0) else "logits_kernel"),
                "algorithmic_bytes_per_launch": lb, "avg_launch_ms": round(logit_avg, 5),
                "stage_ms_in_step": round(logit_step, 5)}
    out = {
        "workload": WORKLOAD_NAMES[cfg], "config_id": cfg, "metric": metric,
        "value": round(job_value(world, keys, ms_per_step, div), 4), "unit": unit,
        "ms_per_step": round(ms_per_step, 5), "rows": rows,
        "timing": mode, "clocks": clk, "roofline": roof,
        "gpu_launches_per_step": step.launches_per_step,
        "l2": ("K pool rotated over three device copies (each step reads pages last read two "
               "steps earlier)" if paged else "256 MB buffer rewritten between steps"),
    }
    if prod:
        out.update({"tokens_per_step": case.T, "k_store_ms": round(logit_avg, 5),
                    "q_quant_ms": round(topk_avg, 5)})
    else:
        # the top-k stage holds the slot map when the step runs the two as
        # one call (paged, the row top-k as its own call)
        with_slots = bool(getattr(step, "_slots_call", 1) is None and paged)
        tb = topk_bytes(case, with_slots)
        tach = tb / (topk_avg * 1e-3) / 1e9
        out.update({
            "keys_scored_per_step": keys,
            "keys_dense_equivalent_per_step": case.keys_scored,
            "logits_ms": round(logit_avg, 5), "topk_ms": round(topk_avg, 5),
            "logits_stage_ms_in_step": round(logit_step, 5),
            "topk_stage_ms_in_step": round(topk_step, 5),
            "topk_rows_per_s": round(world * rows / (topk_avg * 1e-3), 1),
            "topk_roofline": {"stage": ("top-k + slot map (one call)" if with_slots
                                        else "top-k"),
                              "bound": "hbm", "achieved": round(tach, 1), "peak": hbm,
                              "unit": "GB/s", "frac": round(tach / hbm, 4),
                              "algorithmic_bytes_per_launch": tb,
                              "avg_launch_ms": round(topk_avg, 5),
                              "stage_ms_in_step": round(topk_step, 5),
                              "peak_source": f"{src} hbm_gbs"},
            "fused_topk": fused,
        })
    if headline:
        out["_step"] = step
        out["_case"] = case
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    world, rank, local = _dist()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    if args.profile_run:  # warm-up steps only, for ncu captures
        from sparse_attention_indexer_mxfp4_gb300 import (IndexerStep, ProducerStep,
                                                          idx_get_device_status)
        case = _case(args.config, shard=rank)
        step = (ProducerStep(case, device=dev) if _is_producer(case) else
                IndexerStep(case, device=dev, fused_topk=args.fused_topk,
                        fused_slots=not args.split_slots))
        for _ in range(args.warmup):
            step.run()
        torch.cuda.synchronize()
        assert idx_get_device_status() == 0, "device status set during warm-up"
        if rank == 0:
            print(json.dumps({"profile_run": True, "config": args.config,
                              "launches": step.launches_per_step * args.warmup}))
        if world > 1:
            dist.destroy_process_group()
        return

    head = measure(args.config, args, dev, world, rank, headline=True)
    step, case = head.pop("_step"), head.pop("_case")
    e2e = run_e2e(step, case, args, dev) if rank == 0 else None
    per_config = {}
    if not args.no_per_config:
        for c in sorted(WORKLOAD_NAMES):
            if c != args.config:
                r = measure(c, args, dev, world, rank, headline=False)
                per_config[str(c)] = r
                del r
                torch.cuda.empty_cache()
    prod = _is_producer(case)
    out = {
        "metric": head["metric"], "value": head["value"], "unit": head["unit"],
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("bf16 -> e2m1 (e8m0 block scales)" if prod else
                  "e4m3 x e4m3 -> f32" if case.fmt == 0 else
                  "e2m1 x e2m1 (e8m0 block scales) -> f32"),
        "data": "synthetic (seeded; shapes and distributions of the workload description)",
        "config": {"workload": head["workload"], "config_id": args.config, "rows": head["rows"],
                   "keys_scored_per_step": head.get("keys_scored_per_step"),
                   "keys_dense_equivalent_per_step": head.get("keys_dense_equivalent_per_step"),
                   "l2": head["l2"], "timing": head["timing"]},
        "logits_ms" if not prod else "k_store_ms": head.get("logits_ms", head.get("k_store_ms")),
        "topk_ms" if not prod else "q_quant_ms": head.get("topk_ms", head.get("q_quant_ms")),
        "topk_rows_per_s": head.get("topk_rows_per_s"),
        "roofline": head["roofline"],
        "topk_roofline": head.get("topk_roofline"),
        "clocks": head["clocks"],
        "gpu_launches": head["gpu_launches_per_step"] * args.steps,
        "fused_topk": head.get("fused_topk", False),
        "e2e": e2e,
        "per_config": per_config,
    }
    if rank == 0:
        out["cpu_baseline"] = cpu_baseline(case, args) if world == 1 and not args.no_cpu else None
        print(json.dumps(out))
    if world > 1:
        dist.destroy_process_group()


def time_steps_graph(steps, K, flush, clock_soak_s=0.4):
    """K steps captured into one CUDA graph; the timed region is one replay.
    Step i runs buffer set i % len(steps).
    The step time is the replay's time / K from a graph with no event inside
    it: an event node between two kernels cuts the programmatic overlap of
    the second kernel's launch with the end of the first (measured: 8 us a
    step on the paged FP8 decode).  Only with an L2 flush between steps does
    that graph carry events at the step boundaries, so that the flush stays
    outside the summed step times.  The per-stage times come from a second
    graph whose stages are each bracketed by events.
    Before the timed replay, untimed replays keep the GPU loaded for
    clock_soak_s so the clock samples see the kernels running.  Returns None
    if this torch cannot record timing events inside a graph."""
    import torch
    try:
        bounds = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
                  for _ in range(K)]
        evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
               for _ in range(K)]
    except TypeError:
        return None
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())

    def capture(staged):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for i in range(K):
                if flush is not None:
                    flush.fill_(float(i))
                step = steps[i % len(steps)]
                if staged:
                    evs[i][0].record()
                    step.logits_stage()
                    evs[i][1].record()
                    step.topk_stage()
                    evs[i][2].record()
                    step.slots_stage()
                    evs[i][3].record()
                elif flush is not None:
                    bounds[i][0].record()
                    step.run()
                    bounds[i][1].record()
                else:
                    step.run()
        torch.cuda.synchronize()
        g.replay()  # the first replay uploads the graph
        torch.cuda.synchronize()
        return g

    g_step, g_stages = capture(False), capture(True)

    # per-launch time of each stage in steady state: K launches of the stage
    # alone, back to back (rotating buffer sets), events only at the ends, so
    # each launch overlaps the end of the one before as it does in a step
    loop_ms = {}
    if flush is None:
        for name in ("logits_stage", "topk_stage"):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for i in range(K):
                    getattr(steps[i % len(steps)], name)()
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(side):
                e0.record()
                g.replay()
                e1.record()
            torch.cuda.synchronize()
            loop_ms[name] = e0.elapsed_time(e1) / K
    t_end = time.time() + clock_soak_s
    while time.time() < t_end:
        g_step.replay()
        torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(side):
        a.record()
        g_step.replay()
        b.record()
    torch.cuda.synchronize()
    step_ms = [e[0].elapsed_time(e[1]) for e in bounds] if flush is not None else []
    total = a.elapsed_time(b)
    g_stages.replay()
    torch.cuda.synchronize()
    logit_ms = [e[0].elapsed_time(e[1]) for e in evs]
    topk_ms = [e[1].elapsed_time(e[2]) for e in evs]
    ms = sum(step_ms) / K if flush is not None else total / K
    return ms, logit_ms, topk_ms, loop_ms, (
        "cuda graph of the K steps, one replay; stage times in the step from a second replay "
        "with events between the stages; per-launch stage times from graphs of K back-to-back "
        "launches of each stage")


def time_steps_eager(steps, K, flush):
    import torch
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for i in range(K):
        step = steps[i % len(steps)]
        if flush is not None:
            flush.fill_(float(i))
        ev[i][0].record(stream)
        step.logits_stage()
        ev[i][1].record(stream)
        step.topk_stage()
        ev[i][2].record(stream)
        step.slots_stage()
        ev[i][3].record(stream)
    torch.cuda.synchronize()
    logit_ms = [e[0].elapsed_time(e[1]) for e in ev]
    topk_ms = [e[1].elapsed_time(e[2]) for e in ev]
    step_ms = [e[0].elapsed_time(e[3]) for e in ev]
    return sum(step_ms) / K, logit_ms, topk_ms, {}, "eager launches"


def run_e2e(step, case, args, dev):
    """Same metric through the public API with host buffers: each step copies
    the step's inputs (step.input_names(): queries, weights, lengths, block
    table, candidates; for the producers the new keys, queries, weights,
    positions and slots) from pinned host memory and reads its results back
    (step.results(): top-k indices and ragged slots; the quantised queries,
    their scales and weights).  The K cache and the model constants are
    resident device state, not per-step inputs.  Steps run as a serving loop runs them:
    two sets of device buffers; step i's inputs are copied in on one stream
    while step i-1 computes on a second and step i-2's results are copied out
    on a third, each set's copy-in -> compute -> copy-out -> next copy-in
    ordered by stream dependencies.  The K steps (copies and kernels) are
    captured into one CUDA graph, so that, as in the device-timed graph, a
    step's first kernel may start while the step before finishes; the timed
    region is one replay of it, from the first copy-in to the last
    copy-out."""
    import torch

    from sparse_attention_indexer_mxfp4_gb300.synth import PagedCase
    # two buffer sets; paged sets hold their own copy of the K pool, so a
    # step never reads pages the step before it left in L2
    sets = [step, step.twin(kv_copy=isinstance(case, PagedCase))]
    host = {n: getattr(step, n).cpu().pin_memory() for n in step.input_names()}
    outs = [st.results() for st in sets]
    host_out = [[o.cpu().pin_memory() for o in os_] for os_ in outs]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    steps = max(3, args.steps)

    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    for st in sets:  # first launches (library set-up) outside the capture
        with torch.cuda.stream(cap):
            st.run()
    torch.cuda.synchronize()
    copy_in, comp, copy_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def issue(i, h2d_done, comp_done, d2h_done):
        s = i % 2
        st = sets[s]
        with torch.cuda.stream(copy_in):
            if i >= 2:
                copy_in.wait_event(comp_done[i - 2])  # step i-2 has read this set's inputs
            for n, t in host.items():
                getattr(st, n).copy_(t, non_blocking=True)
            h2d_done[i].record(copy_in)
        with torch.cuda.stream(comp):
            comp.wait_event(h2d_done[i])
            if i >= 2:
                comp.wait_event(d2h_done[i - 2])  # step i-2's results are out of this set
            st.run()
            comp_done[i].record(comp)
        with torch.cuda.stream(copy_out):
            copy_out.wait_event(comp_done[i])
            for h, o in zip(host_out[s], outs[s]):
                h.copy_(o, non_blocking=True)
            d2h_done[i].record(copy_out)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        for x in (copy_in, comp, copy_out):
            x.wait_stream(cap)
        evs = [[torch.cuda.Event() for _ in range(steps)] for _ in range(3)]
        for i in range(steps):
            issue(i, *evs)
        for x in (copy_in, comp, copy_out):
            cap.wait_stream(x)
    torch.cuda.synchronize()
    g.replay()  # the first replay uploads the graph
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cap):
        a.record()
        g.replay()
        b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    for h0, h1 in zip(host_out[0], host_out[1]):  # both sets computed the same step
        assert torch.equal(h0, h1), "the two buffer sets returned different results"
    _, unit, div = _metric_unit_div(case)
    return {"value": round(_work(case) / (ms * 1e-3) / div, 4), "unit": unit,
            "ms_per_step": round(ms, 5), "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h),
            "pipeline": "two buffer sets; copy-in, compute and copy-out on three streams, "
                        "the K steps captured into one CUDA graph (copies included)"}


def _oracle_sample(case, nseq, nthreads=0):
    """The oracle's step (logits, mask, top-k, slots) over the first nseq
    sequences (paged) or rows (contiguous) of the workload, or its producers
    over the first nseq tokens; returns the units of work (keys, tokens)."""
    import oracle
    from sparse_attention_indexer_mxfp4_gb300.synth import PagedCase
    if _is_producer(case):
        import torch
        n = nseq

        def bits(x):
            return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).view(
                torch.int16).numpy().view(np.uint16)
        pages = np.zeros((case.num_pages, case.page_stride), np.uint8)
        oracle.k_norm_rope_store(case.fmt, bits(case.k_pre[:n]), case.positions[:n], case.cos_sin,
                                 case.rope_dim, case.norm_weight, case.eps, pages,
                                 case.page_size, case.slots[:n])
        oracle.q_rope_quant(case.fmt, bits(case.q[:n]), case.positions[:n], case.cos_sin,
                            case.rope_dim, case.weights[:n], case.weight_scale)
        return n
    if isinstance(case, PagedCase):
        rows = np.arange(nseq * case.next_n)
        ctx = case.context_lens[rows] if case.ctx_per_row else case.context_lens[:nseq]
        out, _ = oracle.paged_mqa_logits(case.fmt, case.q[rows],
                                         None if case.q_scale is None else case.q_scale[rows],
                                         case.weights[rows], case.pages, case.page_stride,
                                         case.num_pages, case.block_table[:nseq], ctx,
                                         case.ctx_per_row, None, nseq, case.next_n, case.H,
                                         case.D, case.page_size, case.width, nthreads=nthreads)
        ke = np.clip(case.row_ends()[rows], 0, case.width).astype(np.int32)
        if case.cand is not None:
            oracle.apply_candidate_mask(out, None, ke, case.cand[rows], case.cand_block,
                                        nthreads=nthreads)
        out = np.where(np.isnan(out), -np.inf, out)
        idx = oracle.topk(out, ke, case.topk, nthreads=nthreads)
        oracle.topk_to_ragged_slots(idx, case.block_table[:nseq], case.page_size,
                                    case.num_pages, next_n=case.next_n)
        if getattr(case, "source_block", 0):
            bs = case.source_block
            bm = oracle.block_max(out, None, ke, bs)
            oracle.topk(bm, ((ke + bs - 1) // bs).astype(np.int32), case.source_cands)
        return int(ke.sum())
    rows = np.arange(nseq)
    out = oracle.mqa_logits(case.fmt, case.q[rows], None, case.weights[rows], case.k,
                            case.k_scale, case.ks[rows], case.ke[rows], nseq, case.N, case.H,
                            case.D, nthreads=nthreads)
    oracle.topk(out, case.ke[rows], case.topk, nthreads=nthreads)
    return int(np.maximum(case.ke[rows] - case.ks[rows], 0).sum())


def _units(case):
    from sparse_attention_indexer_mxfp4_gb300.synth import PagedCase
    if _is_producer(case):
        return case.T
    return case.B if isinstance(case, PagedCase) else case.M


def cpu_baseline(case, args, target_s: float = 10.0):
    """The oracle as it stands, on this host's cores, over a growing prefix
    of the workload until about target_s seconds of work."""
    import oracle
    n = 1
    total = _units(case)
    while True:
        t = time.time()
        keys = _oracle_sample(case, n)
        dt = time.time() - t
        if dt >= target_s or n >= total:
            break
        n = min(total, max(n + 1, int(n * min(8.0, target_s / max(dt, 1e-3)))))
    _, unit, div = _metric_unit_div(case)
    if _is_producer(case):
        what = (f"first {n} of {total} tokens: fp64 scalar norm + RoPE + quantise of the key "
                f"and of the {case.H} query heads, {dt:.1f} s")
    else:
        what = (f"first {n} of {total} {'sequences' if hasattr(case, 'B') else 'rows'} "
                f"({keys} keys): fp64 scalar logits + mask + top-k + slots, {dt:.1f} s")
    # the single-thread oracle on the whole small contiguous workload
    c1 = _case(1)
    t = time.time()
    k1 = _oracle_sample(c1, c1.M, nthreads=1)
    dt1 = time.time() - t
    return {"value": round(keys / dt / div, 6), "unit": unit, "cores": oracle.default_threads(),
            "kind": "oracle", "sample": what,
            "single_thread": {"workload": WORKLOAD_NAMES[1], "value": round(k1 / dt1 / 1e9, 6),
                              "unit": "Gkeys/s", "seconds": round(dt1, 3), "cores": 1,
                              "sample": f"all {c1.M} rows ({k1} keys): logits + top-k"}}


def run_reference(args):
    world, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    from sparse_attention_indexer_mxfp4_gb300.synth import PagedCase
    case = _case(args.config)
    cores = oracle.default_threads()
    # enough sequences (rows) that the oracle's row threads cover every core
    per = case.next_n if isinstance(case, PagedCase) else 1
    nseq = min(_units(case), max(1, -(-cores // per)))
    for _ in range(args.warmup):
        _oracle_sample(case, nseq)
    t = time.time()
    keys = 0
    for _ in range(args.steps):
        keys += _oracle_sample(case, nseq)
    dt = time.time() - t
    metric, unit, div = _metric_unit_div(case)
    v = keys / dt / div
    total = _units(case)
    print(json.dumps({
        "impl": "reference", "metric": metric, "value": round(v, 6), "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (scalar CPU oracle)",
        "data": "synthetic", "config": {"workload": WORKLOAD_NAMES[args.config],
                                        "config_id": args.config},
        "cpu_baseline": {"value": round(v, 6), "unit": unit, "cores": cores,
                         "kind": "oracle",
                         "sample": f"each step: the first {nseq} of {total} units of the "
                                   f"workload ({keys // max(args.steps, 1)} units of work)"},
        "e2e": {"value": round(v, 6), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}))


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5, 6, 7])
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    p.add_argument("--no-per-config", action="store_true",
                   help="measure the headline workload only")
    p.add_argument("--profile-run", action="store_true",
                   help="run the warm-up steps only and exit (a short command for ncu captures)")
    p.add_argument("--fused-topk", action="store_true",
                   help="paged workloads without a candidate list: one call for the logits and "
                        "the row top-k (idx_paged_mqa_logits_topk)")
    p.add_argument("--split-slots", action="store_true",
                   help="paged workloads: the row top-k and the slot map as two calls "
                        "(idx_topk, idx_topk_to_ragged_slots) instead of idx_topk_ragged_slots")
    args = p.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
