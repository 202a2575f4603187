"""Summaries of the persistent kernel's task trace (MOE_OPT_TRACE).

``MoELayer.trace()`` returns one record per executed task -- the CTA (the
leader of the CTA pair that ran it), the task id, and the %globaltimer times
at which the task was claimed, started and finished -- plus one record per
plan phase and one exit record per pair.
``summarize`` turns those records into what explains a layer's time: each
task type's window and durations, the CTAs' utilisation over time per task
type, the gaps between consecutive tasks on a CTA, and the plan's phases.

Pure host code on numpy arrays; it reads nothing from the device.
"""
from __future__ import annotations

import numpy as np

# task types of the trace (the task id's top four bits)
TYPES = {1: "route", 2: "gather", 3: "gateup", 4: "down", 5: "combine"}
PLAN = 6
EXIT_TASK = 0x7FFFFFFF


def summarize(tr: dict, n_bins: int = 20) -> dict:
    """Summary of one forward's trace.

    ``tr`` holds equal-length arrays ``cta``, ``task``, ``t_claim``,
    ``t_start`` and ``t_end`` (the dict ``MoELayer.trace`` returns).  Times in
    the result are microseconds from the first claim.  Keys:

    - ``span_us``: first claim to last task end;
    - ``grid``: workers (CTA pairs, whose leaders write the records) that
      wrote an exit record;
    - ``types``: per task type, count, first start, last end and the median
      and maximum duration;
    - ``busy_us``: the summed task time divided by the workers (the span the
      tasks would take packed perfectly);
    - ``bins``: ``n_bins`` equal time windows, each with the fraction of
      CTA-time spent in each task type and in total;
    - ``gaps``: count, median and 90th percentile of the idle time between
      consecutive tasks of one CTA, and their sum over the grid;
    - ``plan_phases_us``: the plan's phase boundaries (empty without a plan).
    """
    task = np.asarray(tr["task"], dtype=np.int64)
    cta = np.asarray(tr["cta"], dtype=np.int64)
    t_claim = np.asarray(tr["t_claim"], dtype=np.int64)
    t_start = np.asarray(tr["t_start"], dtype=np.int64)
    t_end = np.asarray(tr["t_end"], dtype=np.int64)
    is_exit = task == EXIT_TASK
    kind = np.where(is_exit, 0, task >> 28)
    real = ~is_exit & (kind >= 1) & (kind <= 5)
    if not real.any():
        return {"span_us": 0.0, "grid": int(is_exit.sum()), "types": {}, "busy_us": 0.0,
                "bins": [], "gaps": {"n": 0}, "plan_phases_us": []}
    t0 = t_claim[real].min()
    start = (t_start - t0) / 1e3
    end = (t_end - t0) / 1e3
    grid = int(is_exit.sum()) or int(np.unique(cta[real]).size)
    span = float(end[real].max())

    types = {}
    for k, name in TYPES.items():
        sel = real & (kind == k)
        if sel.any():
            dur = end[sel] - start[sel]
            types[name] = {"n": int(sel.sum()), "start_us": float(start[sel].min()),
                           "end_us": float(end[sel].max()),
                           "median_us": float(np.median(dur)), "max_us": float(dur.max())}
    busy = float(np.sum(end[real] - start[real]) / grid)

    bins = []
    edges = np.linspace(0.0, span, n_bins + 1)
    for a, b in zip(edges[:-1], edges[1:]):
        width = max(b - a, 1e-9)
        overlap = np.clip(np.minimum(end, b) - np.maximum(start, a), 0.0, None)
        row = {"from_us": float(a), "to_us": float(b)}
        total = 0.0
        for k, name in TYPES.items():
            frac = float(overlap[real & (kind == k)].sum() / (grid * width))
            row[name] = frac
            total += frac
        row["total"] = total
        bins.append(row)

    idx = np.where(real)[0]
    idx = idx[np.lexsort((start[idx], cta[idx]))]
    same = cta[idx][1:] == cta[idx][:-1]
    gap = (start[idx][1:] - end[idx][:-1])[same]
    gaps = {"n": int(gap.size)}
    if gap.size:
        gaps.update(median_us=float(np.median(gap)), p90_us=float(np.percentile(gap, 90)),
                    sum_over_grid_us=float(gap.sum() / grid))

    plan = ~is_exit & (kind == PLAN)
    phases = sorted(float(end[i]) for i in np.where(plan)[0])
    return {"span_us": span, "grid": grid, "types": types, "busy_us": busy, "bins": bins,
            "gaps": gaps, "plan_phases_us": phases}


def format_summary(s: dict) -> str:
    """The summary as a few lines of text."""
    lines = [f"span {s['span_us']:.1f} us, grid {s['grid']}, "
             f"busy {s['busy_us']:.1f} us per CTA"]
    for name, t in s["types"].items():
        lines.append(f"  {name:8s} n={t['n']:6d}  {t['start_us']:8.1f} .. {t['end_us']:8.1f} us"
                     f"  median {t['median_us']:7.2f}  max {t['max_us']:7.2f}")
    for b in s["bins"]:
        parts = " ".join(f"{n}:{b[n]:.2f}" for n in TYPES.values())
        lines.append(f"  [{b['from_us']:8.1f}, {b['to_us']:8.1f}) util {b['total']:.2f}  {parts}")
    g = s["gaps"]
    if g.get("n"):
        lines.append(f"  gaps: n={g['n']} median {g['median_us']:.2f} us, p90 {g['p90_us']:.2f} us, "
                     f"{g['sum_over_grid_us']:.1f} us per CTA")
    if s["plan_phases_us"]:
        lines.append("  plan phases (us): " + " ".join(f"{v:.1f}" for v in s["plan_phases_us"]))
    return "\n".join(lines)
