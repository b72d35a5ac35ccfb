"""Kernel timeline analysis of the records that ``fs_trace_read`` returns.

Each record is one block of one kernel launch: its tag, whether it passed
its wait for the preceding kernel, its SM, its block index and three
%globaltimer stamps (entry, after the wait, end). A block that passed the
wait did so only after every block of the preceding launch had finished, so
ordering the waiting blocks by the time they passed it orders the launches;
consecutive launches of a decode step never share a tag, so a run of one tag
in that order is one launch. Blocks that left without waiting (attention
splits past a lane's length) do no work and are left out.

Per launch: ``gap`` = first wait passed - previous launch's last block end
(dependency resolution: the predecessor's completion becoming visible),
``body`` = last block end - first wait passed, ``contribution`` = gap + body
(the launch's share of the step's wall time), ``ahead`` = first wait passed -
first block entry (how early programmatic dependent launch brought it in).
"""
from __future__ import annotations

from collections import OrderedDict

import numpy as np

from .fs import TRACE_TAGS


def decode(recs: np.ndarray) -> dict:
    w0 = recs[:, 0].astype(np.uint64)
    return {"tag": (w0 >> np.uint64(40)).astype(np.int64),
            "waited": ((w0 >> np.uint64(39)) & np.uint64(1)).astype(bool),
            "sm": ((w0 >> np.uint64(24)) & np.uint64(0x7fff)).astype(np.int64),
            "block": (w0 & np.uint64(0xffffff)).astype(np.int64),
            "t_entry": recs[:, 1].astype(np.int64),
            "t_ready": recs[:, 2].astype(np.int64),
            "t_exit": recs[:, 3].astype(np.int64)}


def launches(recs: np.ndarray) -> list:
    """Launches in stream order: dicts of tag, name, blocks, first_entry,
    first_ready, last_exit (ns)."""
    d = decode(recs)
    idx = np.nonzero(d["waited"])[0]
    idx = idx[np.argsort(d["t_ready"][idx], kind="stable")]
    out = []
    for i in idx:
        tag = int(d["tag"][i])
        if not out or out[-1]["tag"] != tag:
            out.append({"tag": tag, "name": TRACE_TAGS.get(tag, str(tag)), "blocks": 0,
                        "first_entry": int(d["t_entry"][i]), "first_ready": int(d["t_ready"][i]),
                        "last_exit": int(d["t_exit"][i])})
        L = out[-1]
        L["blocks"] += 1
        L["first_entry"] = min(L["first_entry"], int(d["t_entry"][i]))
        L["last_exit"] = max(L["last_exit"], int(d["t_exit"][i]))
    return out


def summarize(recs: np.ndarray, steps: int) -> dict:
    """Per kernel name: launches per step and mean gap / body / contribution /
    ahead in microseconds, plus the traced span per step. The first launch
    (no traced predecessor) is left out of the means."""
    ls = launches(recs)
    agg = OrderedDict()
    for prev, cur in zip(ls, ls[1:]):
        a = agg.setdefault(cur["name"], {"n": 0, "gap": 0.0, "body": 0.0, "ahead": 0.0})
        a["n"] += 1
        a["gap"] += (cur["first_ready"] - prev["last_exit"]) / 1e3
        a["body"] += (cur["last_exit"] - cur["first_ready"]) / 1e3
        a["ahead"] += (cur["first_ready"] - cur["first_entry"]) / 1e3
    span = (ls[-1]["last_exit"] - ls[0]["last_exit"]) / 1e3 if len(ls) > 1 else 0.0
    kern = {}
    for name, a in sorted(agg.items(), key=lambda kv: -(kv[1]["gap"] + kv[1]["body"])):
        n = a["n"]
        kern[name] = {"launches_per_step": n / max(1, steps),
                      "mean_gap_us": a["gap"] / n, "mean_body_us": a["body"] / n,
                      "mean_ahead_us": a["ahead"] / n,
                      "share": (a["gap"] + a["body"]) / span if span else None}
    return {"launches": len(ls), "steps": steps,
            "us_per_step": span / max(1, steps) if len(ls) > 1 else None,
            "kernels": kern}


def table(summary: dict) -> str:
    lines = [f"{'kernel':14s} {'per step':>8s} {'gap us':>8s} {'body us':>8s} "
             f"{'ahead us':>8s} {'share':>6s}"]
    for name, k in summary["kernels"].items():
        lines.append(f"{name:14s} {k['launches_per_step']:8.1f} {k['mean_gap_us']:8.2f} "
                     f"{k['mean_body_us']:8.2f} {k['mean_ahead_us']:8.2f} "
                     f"{100 * (k['share'] or 0):5.1f}%")
    lines.append(f"traced span per step: {summary['us_per_step']:.1f} us over "
                 f"{summary['launches']} launches")
    return "\n".join(lines)
