"""Turn a step timeline (``Engine.read_trace()``) into per-phase and per-SM figures.

Each consumer event covers one tile or queue item: when its first operand chunk
had landed in shared memory (start), when its dependency counter was satisfied
(met) and when it finished (end), in globaltimer nanoseconds.  Producer events
record how long each SM's producer waited for routing before it could stream
expert weights.
"""
from __future__ import annotations

import numpy as np

OPS = {1: "embed", 2: "qkv", 3: "attn", 4: "oproj", 5: "router", 6: "moe", 7: "head", 100: "gate_up", 101: "down"}


def events(tr: np.ndarray):
    """Flatten to a structured array: cta, t_start, t_met, t_end, op, layer, kind, idx, producer."""
    rows = []
    n_ctas, cap, _ = tr.shape
    for c in range(n_ctas):
        nc = int(tr[c, 0, 0])
        npv = int(tr[c, 0, 2])
        for i in range(1, min(nc, cap // 2)):
            rows.append((c, *tr[c, i, :3], int(tr[c, i, 3]), 0))
        for j in range(min(npv, cap // 2)):
            rows.append((c, *tr[c, cap - 1 - j, :3], int(tr[c, cap - 1 - j, 3]), 1))
    dt = np.dtype([("cta", "i4"), ("t0", "u8"), ("tm", "u8"), ("t1", "u8"), ("tag", "u8"), ("prod", "i4")])
    a = np.array(rows, dtype=dt)
    return a


def summarize(tr: np.ndarray, n_layers: int) -> dict:
    """Per-phase windows (first start .. last end, relative to kernel start), mean wait
    per tile, and the share of consumer time spent waiting on dependencies."""
    ev = events(tr)
    t_kernel = int(min(tr[c, 0, 1] for c in range(tr.shape[0]) if tr[c, 0, 1]))
    op = (ev["tag"] & 0xff).astype(int)
    layer = ((ev["tag"] >> 8) & 0xffff).astype(int)
    out = {"phases": [], "wait_share": None, "step_us": None}
    kind = ((ev["tag"] >> 24) & 0xff).astype(int)
    chunks = ev[(ev["prod"] == 0) & (kind == 4)]
    out["marks"] = ev[(ev["prod"] == 0) & (kind == 5)]
    ev = ev[~((ev["prod"] == 0) & ((kind == 4) | (kind == 5)))]
    op = (ev["tag"] & 0xff).astype(int)
    layer = ((ev["tag"] >> 8) & 0xffff).astype(int)
    if len(chunks):
        cop = (chunks["tag"] & 0xff).astype(int)
        out["chunks"] = {}
        for o in sorted(set(cop.tolist())):
            cc = chunks[cop == o]
            lat = (cc["tm"].astype(np.int64) - cc["t0"].astype(np.int64)) / 1e3
            hold = (cc["t1"].astype(np.int64) - cc["tm"].astype(np.int64)) / 1e3
            out["chunks"][OPS.get(o, str(o))] = dict(n=int(len(cc)), issue_to_seen_us_median=float(np.median(lat)),
                                                    issue_to_seen_us_p90=float(np.percentile(lat, 90)),
                                                    seen_to_release_us_median=float(np.median(hold)))
    cons = ev[ev["prod"] == 0]
    if len(cons) == 0:
        return out
    t_end = int(cons["t1"].max())
    out["step_us"] = (t_end - t_kernel) / 1e3
    busy = (cons["t1"] - cons["tm"]).astype(np.int64).sum()
    wait = (cons["tm"] - cons["t0"]).astype(np.int64).sum()
    out["wait_share"] = float(wait / max(1, wait + busy))
    for l in list(range(n_layers)) + [n_layers]:
        for o in (1, 2, 3, 4, 5, 6, 7):
            sel = (ev["prod"] == 0) & (op == o) & ((layer == l) | ((o == 1) & (l == 0)))
            if o == 7 and l != n_layers:
                continue
            if not sel.any():
                continue
            e = ev[sel]
            out["phases"].append(dict(layer=l, op=OPS[o], n=int(sel.sum()),
                                      start_us=(int(e["t0"].min()) - t_kernel) / 1e3,
                                      met_us=(int(e["tm"].max()) - t_kernel) / 1e3,
                                      end_us=(int(e["t1"].max()) - t_kernel) / 1e3,
                                      mean_wait_us=float((e["tm"] - e["t0"]).astype(np.int64).mean() / 1e3),
                                      mean_work_us=float((e["t1"] - e["tm"]).astype(np.int64).mean() / 1e3)))
        selp = (ev["prod"] == 1) & (layer == l)
        if selp.any():
            e = ev[selp]
            out["phases"].append(dict(layer=l, op="route_wait(producer)", n=int(selp.sum()),
                                      start_us=(int(e["t0"].min()) - t_kernel) / 1e3,
                                      met_us=(int(e["tm"].max()) - t_kernel) / 1e3,
                                      end_us=(int(e["tm"].max()) - t_kernel) / 1e3,
                                      mean_wait_us=float((e["tm"] - e["t0"]).astype(np.int64).mean() / 1e3),
                                      mean_work_us=0.0))
    return out


def format_summary(s: dict, layers=(0, 1, 24)) -> str:
    lines = [f"step {s['step_us']:.1f} us; consumer time waiting on dependencies {100 * s['wait_share']:.1f}%"]
    for k, v in s.get("chunks", {}).items():
        lines.append(f"  chunks {k:>8}: n {v['n']:6d}  issue->seen median {v['issue_to_seen_us_median']:7.2f} us "
                     f"(p90 {v['issue_to_seen_us_p90']:7.2f})  seen->release median {v['seen_to_release_us_median']:6.2f} us")
    lines.append(f"{'layer':>5} {'phase':>22} {'n':>5} {'start':>9} {'met(max)':>9} {'end':>9} {'wait':>7} {'work':>7}")
    for ph in s["phases"]:
        if ph["layer"] in layers or ph["op"] in ("head", "embed"):
            lines.append(f"{ph['layer']:>5} {ph['op']:>22} {ph['n']:>5} {ph['start_us']:>9.1f} {ph['met_us']:>9.1f} "
                         f"{ph['end_us']:>9.1f} {ph['mean_wait_us']:>7.2f} {ph['mean_work_us']:>7.2f}")
    return "\n".join(lines)
