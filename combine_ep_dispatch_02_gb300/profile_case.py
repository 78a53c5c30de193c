"""A small, bounded run of one phase of the path, for ncu captures.

    python -m combine_ep_dispatch_02_gb300.profile_case --phase combine --tokens-per-rank 1024 --launches 4

runs the DeepSeek-V3-shaped workload (W=8, 32 experts per rank, top-8, hidden 7168 BF16, Zipf
routing, FP32 weights, identity expert) at the given tokens per rank, sets up whatever the phase
needs (a dispatch before a combine, a quantised wire before a wire combine), then launches the
phase `--launches` times back to back.  At 1024 tokens per rank the device holds about 1.2 GB
(plan, inputs, outputs; 1.7 GB for the wire phases), and every phase but routing reads or
writes more than the 129 MB L2, so DRAM counters mean what they do at full size.  An ncu
command selects the phase's kernel by name, skips the warm-up launches (-s) and captures one to
three (-c); the setup's own launches of other kernels (and the routing launch before each
scatter) are not selected.

Phases and their kernels:
    route            ep_route_kernel
    scatter          ep_scatter_kernel               (BF16 rows)
    scatter_fp8      ep_scatter_quant_kernel         (quantising dispatch to FP8 e4m3)
    scatter_fp4      ep_scatter_quant_fp4_kernel     (quantising dispatch to MX FP4)
    combine          ep_combine_kernel
    quantise_fp8     ep_quantise_rows_kernel         (expert rows to the FP8 wire)
    quantise_fp4     ep_quantise_rows_fp4_kernel     (expert rows to the MX FP4 wire)
    combine_fp8      ep_combine_fp8_kernel
    combine_fp4      ep_combine_fp4_kernel
    grouped_route    ep_route_kernel, the form that also numbers the expert-grouped view
    fused_copy       ep_group_from_source_kernel (the fused dispatch's copy into the grouped view)
    ungroup          ep_ungroup_kernel (the grouped view's inverse)

The three grouped phases run the small grouped workload instead (W=4, 64 experts per rank,
top-8, hidden 7168 BF16, uniform routing, --tokens-per-rank 256 by default for them), the regime
the grouped view's kernels are latency-bound in; its grouped view holds 3.8 GB, and each of
these kernels moves 0.13-0.17 GB, inside the L2, so their captures are read for issue and
stall figures rather than DRAM bytes.

Prints one line per run with the phase, the tokens and the algorithmic bytes of one launch of
the phase's kernel, which a traffic figure is compared with.  `--record RUN_JSON NCU_CSV COMMAND`
enters such a capture in profiles/dram_traffic.json with the kernel's code digest, from which
bench.py derives the full-size traffic while the kernel's code is unchanged.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import json
import os
import statistics

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")

PHASES = ("route", "scatter", "scatter_fp8", "scatter_fp4", "combine", "quantise_fp8",
          "quantise_fp4", "combine_fp8", "combine_fp4", "grouped_route", "fused_copy", "ungroup")
GROUPED_PHASES = ("grouped_route", "fused_copy", "ungroup")
# the CUDA source that holds each phase's kernel (its code digest goes beside a recorded figure)
SOURCES = {"route": "ep_route.cu", "scatter": "ep_scatter.cu", "scatter_fp8": "ep_scatter.cu",
           "scatter_fp4": "ep_scatter.cu", "combine": "ep_combine.cu", "quantise_fp8": "ep_fp8wire.cu",
           "quantise_fp4": "ep_fp8wire.cu", "combine_fp8": "ep_fp8wire.cu", "combine_fp4": "ep_fp8wire.cu",
           "grouped_route": "ep_route.cu", "fused_copy": "ep_grouped.cu", "ungroup": "ep_grouped.cu"}


def code_digest(*files) -> str:
    """sha256 of C/CUDA sources with comments and whitespace removed (string and character
    literals kept), so an edit that only touches comments leaves it unchanged."""
    h = hashlib.sha256()
    for f in files:
        text = open(f, encoding="utf-8").read()
        out, i, n = [], 0, len(text)
        while i < n:
            c = text[i]
            if text.startswith("//", i):
                j = text.find("\n", i)
                i = n if j < 0 else j
            elif text.startswith("/*", i):
                j = text.find("*/", i + 2)
                i = n if j < 0 else j + 2
                out.append(" ")
            elif c in "\"'":
                j = i + 1
                while j < n and text[j] != c:
                    j += 2 if text[j] == "\\" else 1
                out.append(text[i:j + 1])
                i = j + 1
            else:
                out.append(c)
                i += 1
        h.update(" ".join("".join(out).split()).encode())
    return h.hexdigest()


def kernel_digest(phase: str) -> str:
    """Code digest of the phase kernel's source file and the shared header it includes."""
    csrc = os.path.join(PKG, "csrc")
    return code_digest(os.path.join(csrc, SOURCES[phase]), os.path.join(csrc, "ep_common.cuh"))


def record(phase: str, run_line: dict, ncu_csv: str, command: str) -> dict:
    """Enter one capture in profiles/dram_traffic.json: the mean DRAM bytes (read + write) per
    captured launch of the phase's kernel, from an ncu --csv log of dram__bytes_read.sum and
    dram__bytes_write.sum, beside the launch's algorithmic bytes and the kernel's code digest."""
    per_launch = {}
    with open(ncu_csv) as f:
        rows = [ln for ln in f if ln.startswith('"')]
    for row in csv.DictReader(rows):
        if row["Metric Name"] in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            v = float(row["Metric Value"].replace(",", ""))
            scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}[row["Metric Unit"]]
            per_launch.setdefault(row["ID"], {})[row["Metric Name"]] = v * scale
    launches = [d for d in per_launch.values() if len(d) == 2]
    if not launches:
        raise ValueError(f"no DRAM metrics in {ncu_csv}")
    read = statistics.mean(d["dram__bytes_read.sum"] for d in launches)
    write = statistics.mean(d["dram__bytes_write.sum"] for d in launches)
    try:
        with open(TRAFFIC_FILE) as f:
            doc = json.load(f)
    except OSError:
        doc = {"about": "ncu DRAM bytes per launch of each kernel on the DeepSeek-V3 shape at a "
                        "reduced token count; bench.py scales traffic / algorithmic bytes to the "
                        "full launch", "kernels": {}}
    doc["kernels"][phase] = {
        "case": f"DeepSeek-V3 shape, {run_line['tokens_per_rank']} tokens per rank "
                f"({run_line['tokens']} tokens, {run_line['token_dest_pairs']} pairs)",
        "command": command, "captured_launches": len(launches),
        "dram_read_bytes_per_launch": int(round(read)), "dram_write_bytes_per_launch": int(round(write)),
        "dram_bytes_per_launch": int(round(read + write)),
        "algorithmic_bytes_per_launch": run_line["kernel_algorithmic_bytes"],
        "traffic_over_algorithmic": round((read + write) / run_line["kernel_algorithmic_bytes"], 4),
        "code_digest": kernel_digest(phase)}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(doc, f, indent=1, sort_keys=True)
        f.write("\n")
    return doc["kernels"][phase]


def kernel_bytes(phase: str, N: int, P: int, W: int, H: int, k: int, entries: int = 0) -> int:
    """Algorithmic bytes of one launch of the phase's kernel (weights given, no caller scales):
    what the kernel must read and write, each byte once.  `entries` counts the grouped view's
    list entries (received rows times their distinct local experts) for the grouped phases."""
    F = min(W, k)
    fp8_row, fp4_row = H + 4 * (H // 128), H // 2 + H // 32
    return {
        "route": N * 4 * k + P * 4,
        "scatter": N * (2 * H + 8 * k) + P * (2 * H + 8 * k),
        "scatter_fp8": N * (2 * H + 8 * k) + P * (fp8_row + 8 * k),
        "scatter_fp4": N * (2 * H + 8 * k) + P * (fp4_row + 8 * k),
        "combine": P * (2 * H + 4 * k) + N * (2 * H + 4 * k) + N * 4 * F,
        "quantise_fp8": P * (2 * H + fp8_row),
        "quantise_fp4": P * (2 * H + fp4_row),
        "combine_fp8": P * (fp8_row + 4 * k) + N * (2 * H + 4 * k) + N * 4 * F,
        "combine_fp4": P * (fp4_row + 4 * k) + N * (2 * H + 4 * k) + N * 4 * F,
        # routing that also writes each entry's list slot (map) and source token (src_info)
        "grouped_route": N * 4 * k + P * 4 + entries * 8,
        # source rows and their index / weight rows read once; a row per entry and the
        # receive rows' index / weight rows written
        "fused_copy": N * (2 * H + 8 * k) + entries * 2 * H + P * 8 * k,
        # the entries' expert outputs read, a row per received row written
        "ungroup": entries * 2 * H + P * (2 * H + 4 * k),
    }[phase]


def run(phase: str, tokens_per_rank: int, launches: int) -> dict:
    import numpy as np
    import torch

    import combine_ep_dispatch_02_gb300 as ep
    from combine_ep_dispatch_02_gb300 import build, workloads

    if phase not in PHASES:
        raise ValueError(f"phase {phase!r} is not one of {PHASES}")
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if phase in GROUPED_PHASES:
        return run_grouped(phase, tokens_per_rank, launches)
    wl = workloads.make_workload("dsv3", max_tok=tokens_per_rank)
    plan_dtype = {"scatter_fp8": "bf16_fp8", "scatter_fp4": "bf16_mxfp4"}.get(phase, "bf16")
    plan = ep.Plan(wl.W, wl.E, wl.k, wl.H, plan_dtype, 0, wl.M, device=dev)
    x = torch.from_numpy(wl.x.view(np.int16)).to(dev)
    idx = torch.from_numpy(wl.indices).to(dev)
    w = torch.from_numpy(wl.weights).to(dev)
    out = torch.empty((wl.W, wl.M, wl.H), dtype=torch.bfloat16, device=dev)
    out_w = torch.empty((wl.W, wl.M, wl.k), dtype=torch.float32, device=dev)
    d = plan.dispatch(x, w, None, idx, wl.n_tok)
    q = sc = None
    if phase in ("combine_fp8", "quantise_fp8"):
        q, sc = plan.quantize_received(d.recv_x, d.epoch)
    elif phase in ("combine_fp4", "quantise_fp4"):
        q, sc = plan.quantize_received_fp4(d.recv_x, d.epoch)
    for _ in range(launches):
        if phase == "route":
            d = plan.dispatch_route(idx, wl.n_tok)
        elif phase.startswith("scatter"):       # a scatter follows the routing of its call
            d = plan.dispatch_route(idx, wl.n_tok)
            plan.dispatch_scatter(x, w, None, idx)
        elif phase == "combine":
            plan.combine(d.recv_x, d.recv_w, d.epoch, out=out, out_w=out_w)
        elif phase == "quantise_fp8":
            plan.quantize_received(d.recv_x, d.epoch, q=q.view(torch.uint8), scales=sc)
        elif phase == "quantise_fp4":
            plan.quantize_received_fp4(d.recv_x, d.epoch, q=q, scales=sc)
        elif phase == "combine_fp8":
            plan.combine_fp8(q, sc, d.recv_w, d.epoch, out=out, out_w=out_w)
        else:
            plan.combine_fp4(q, sc, d.recv_w, d.epoch, out=out, out_w=out_w)
    torch.cuda.synchronize()
    status = plan.status()
    P = int(d.recv_count.sum().item())
    plan.close()
    if status != 0:
        raise RuntimeError(f"device status {status}")
    return {"phase": phase, "tokens_per_rank": wl.M, "tokens": wl.N, "token_dest_pairs": P,
            "launches": launches, "kernel_algorithmic_bytes": kernel_bytes(phase, wl.N, P, wl.W, wl.H, wl.k)}


def run_grouped(phase: str, tokens_per_rank: int, launches: int) -> dict:
    """The grouped phases on the small grouped workload: a fused dispatch into the grouped view
    sets it up; then `launches` fused dispatches (grouped_route, fused_copy) or inverses (ungroup)."""
    import numpy as np
    import torch

    import combine_ep_dispatch_02_gb300 as ep
    from combine_ep_dispatch_02_gb300 import workloads

    dev = torch.device("cuda", 0)
    wl = workloads.make_workload("small", max_tok=tokens_per_rank)
    plan = ep.Plan(wl.W, wl.E, wl.k, wl.H, "bf16", 0, wl.M, device=dev)
    x = torch.from_numpy(wl.x.view(np.int16)).to(dev)
    idx = torch.from_numpy(wl.indices).to(dev)
    w = torch.from_numpy(wl.weights).to(dev)
    d, px, cnt, _, _ = plan.dispatch_grouped(x, w, None, idx, wl.n_tok)
    out = None
    for _ in range(launches):
        if phase == "ungroup":
            out = plan.ungroup_by_expert(px.view(torch.bfloat16), d.epoch, out=out)
        else:
            d, px, cnt, _, _ = plan.dispatch_grouped(x, w, None, idx, wl.n_tok, packed_x=px)
    torch.cuda.synchronize()
    status = plan.status()
    P = int(d.recv_count.sum().item())
    entries = int(cnt.sum().item())
    plan.close()
    if status != 0:
        raise RuntimeError(f"device status {status}")
    return {"phase": phase, "workload": "small", "tokens_per_rank": wl.M, "tokens": wl.N, "token_dest_pairs": P,
            "expert_entries": entries, "launches": launches,
            "kernel_algorithmic_bytes": kernel_bytes(phase, wl.N, P, wl.W, wl.H, wl.k, entries)}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--phase", required=True, choices=PHASES)
    ap.add_argument("--tokens-per-rank", type=int, default=None,
                    help="default 1024 (DeepSeek-V3 shape), 256 for the grouped phases")
    ap.add_argument("--launches", type=int, default=4)
    ap.add_argument("--record", nargs=3, metavar=("RUN_JSON", "NCU_CSV", "COMMAND"),
                    help="enter a capture in profiles/dram_traffic.json instead of running: the "
                         "JSON line a run printed, the ncu --csv log, and the ncu command line")
    a = ap.parse_args()
    if a.record:
        with open(a.record[0]) as f:
            line = json.loads([ln for ln in f if ln.startswith("{")][-1])
        print(json.dumps(record(a.phase, line, a.record[1], a.record[2])), flush=True)
        return
    tpr = a.tokens_per_rank or (256 if a.phase in GROUPED_PHASES else 1024)
    print(json.dumps(run(a.phase, tpr, a.launches)), flush=True)


if __name__ == "__main__":
    main()
