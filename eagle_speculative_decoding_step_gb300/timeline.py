"""Per-kernel timeline of graph-replayed steps, from the instrumented build.

The library built with ``build(timeline=True)`` (libeaglespec_timeline.so,
loaded when EAGLESPEC_TIMELINE=1) has thread 0 of every block record the global
timer at the block's start and exit into a device log (layout in csrc/common.cuh,
"timeline").  This module attaches the log, and turns it into launches (a
kernel's blocks, in start order, grouped by its grid size) and a per-kernel
table of one step: each launch is charged the time from the later of its own
start and the previous launches' last end to its own end (the step's wall time
split along the kernel sequence; programmatic-dependent-launch overlap counts
for the kernel that finishes later).  ``bench.py --timeline FILE`` drives it.
Timings from the instrumented build are for attribution only, not bench values.
"""
import ctypes

import numpy as np

# kernel ids of csrc/common.cuh (enum TLKernel), index = id
NAMES = [None, "tc_kernel (GEMMs, LM head)", "attn_ws_kernel", "attn_mma_kernel", "attn_split_kernel",
         "attn_combine_kernel", "prologue_kernel", "epi_store_kernel", "epi_qkv_kernel", "resnorm_kernel",
         "epi_swiglu_kernel", "simt_gemm_kernel", "row_stats_kernel", "topk_select_kernel", "rescore_kernel",
         "cand_best_kernel", "lm_merge_kernel", "tree_expand_kernel", "verify_greedy_kernel",
         "verify_rejection_kernel", "reject_threshold_kernel", "prefill_inputs_kernel", "spec_metadata_kernel",
         "gather_rows_kernel"]
UNITS = ("layer", "lmhead", "metadata", "prefill", "tc_gemm", "tree", "verify")
SLOTS = 1 << 20
LOG_WORDS = 8 + 4 * SLOTS


def attach(lib, ptr):
    """Point every translation unit's log at device address ptr (0 detaches)."""
    for u in UNITS:
        rc = getattr(lib, "spec_timeline_set_" + u)(ctypes.c_void_p(ptr))
        if rc != 0:
            raise RuntimeError("spec_timeline_set_%s failed (%d)" % (u, rc))


def launches(log):
    """Launches from a log (uint64 / int64 array): list of dicts with start, end
    (ns, global timer), kernel name and block count, sorted by start."""
    raw = np.asarray(log).view(np.uint64)
    n = min(int(raw[0] & 0xffffffff), SLOTS)
    e = raw[8:8 + 4 * n].reshape(n, 4).astype(np.int64)
    kid = e[:, 3] & 0xff
    grid = (e[:, 3] >> 8) & 0xffffff
    out = []
    for k in np.unique(kid):
        sel = np.where(kid == k)[0]
        sel = sel[np.argsort(e[sel, 0], kind="stable")]
        i = 0
        while i < len(sel):
            g = max(1, int(grid[sel[i]]))
            blk = sel[i:i + g]
            ends = e[blk, 2]
            out.append({"start": int(e[blk, 0].min()), "end": int(ends.max()),
                        "tail": int(ends.max() - np.median(ends)),
                        "name": NAMES[int(k)] if int(k) < len(NAMES) else "kernel %d" % k,
                        "blocks": len(blk), "grid": g})
            i += g
    out.sort(key=lambda x: x["start"])
    return out


def last_step(ls):
    """The launches after the second-to-last verifier launch, up to the last."""
    ver = [i for i, l in enumerate(ls) if l["name"].startswith("verify_")]
    if len(ver) < 2:
        return ls
    return ls[ver[-2] + 1:ver[-1] + 1]


def attribute(step):
    """Per kernel: launches, summed launch durations, and the charged wall time."""
    if not step:
        return {}, 0.0
    t0 = step[0]["start"]
    prev = t0
    per = {}
    for l in step:
        charged = max(0, l["end"] - max(prev, l["start"]))
        prev = max(prev, l["end"])
        d = per.setdefault(l["name"], {"launches": 0, "dur_ns": 0, "charged_ns": 0, "tail_ns": 0})
        d["launches"] += 1
        d["dur_ns"] += l["end"] - l["start"]
        d["charged_ns"] += charged
        d["tail_ns"] += l.get("tail", 0)
    return per, (prev - t0)


def markdown(step):
    """Table of one step's kernels, largest charged time first."""
    per, span = attribute(step)
    lines = ["| kernel | launches | charged us | share | mean launch us (start to end) | mean tail us |",
             "|---|---|---|---|---|---|"]
    for name, d in sorted(per.items(), key=lambda x: -x[1]["charged_ns"]):
        lines.append("| `%s` | %d | %.1f | %.1f %% | %.1f | %.1f |" % (
            name, d["launches"], d["charged_ns"] / 1e3, 100.0 * d["charged_ns"] / max(span, 1),
            d["dur_ns"] / d["launches"] / 1e3, d["tail_ns"] / d["launches"] / 1e3))
    lines.append("")
    lines.append("Step span (first launch start to last end): %.1f us, %d launches.  Tail: a launch's last "
                 "block end minus its median block end (for the one-block-per-SM GEMMs, how much the slowest "
                 "SM's share lags)." % (span / 1e3, len(step)))
    return "\n".join(lines)


def sequence(step):
    """One line per launch: start, end (us from the step's first start), duration, tail, name, blocks."""
    if not step:
        return ""
    t0 = step[0]["start"]
    return "\n".join("%9.1f %9.1f %8.1f %6.1f  %-28s %d" % (
        (l["start"] - t0) / 1e3, (l["end"] - t0) / 1e3, (l["end"] - l["start"]) / 1e3, l.get("tail", 0) / 1e3,
        l["name"], l["blocks"]) for l in step)
