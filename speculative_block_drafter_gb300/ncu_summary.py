"""Summarise an ncu launch list (``--metrics gpu__time_duration.sum --csv``) per kernel.

    python -m speculative_block_drafter_gb300.ncu_summary launches.csv [--after NAME] [--step-launches N]

Prints, per kernel name (template arguments kept, parameter list dropped), the
number of launches, the total device time and its share of the total. With
``--after`` and ``--step-launches`` it also cuts out one step: the last
complete window of N of the library's launches that follows a launch whose
name begins with NAME (the step's last kernel), and prints the same table. ncu serialises launches and runs each
one cold, so the absolute times are longer than in a graph replay; the shares
are what compare.
"""
from __future__ import annotations

import argparse
import collections
import csv
import re


def read(path):
    with open(path, newline="") as f:
        rows = list(csv.reader(f))
    head = next(i for i, r in enumerate(rows) if r and r[0] == "ID")
    h = rows[head]
    ki, vi, ui = h.index("Kernel Name"), h.index("Metric Value"), h.index("Metric Unit")
    gi = h.index("Grid Size")
    out = []
    for r in rows[head + 1:]:
        if len(r) <= vi or not r[vi]:
            continue
        name = re.sub(r"\(.*", "", r[ki]).replace("dfl::", "").strip()
        name = re.sub(r"^void ", "", name)
        t = float(r[vi].replace(",", ""))
        unit = r[ui]
        t_us = t / 1e3 if unit == "ns" else (t if unit == "us" else t * 1e3 if unit == "ms" else t)
        out.append((name, t_us, r[gi]))
    return out


def table(launches, title):
    agg = collections.OrderedDict()
    for name, t, _ in launches:
        a = agg.setdefault(name, [0, 0.0])
        a[0] += 1
        a[1] += t
    total = sum(a[1] for a in agg.values())
    lines = [f"### {title}", "", f"{len(launches)} launches, {total:.1f} us of device time", "",
             "| kernel | launches | total us | share |", "|---|---:|---:|---:|"]
    for name, (n, t) in sorted(agg.items(), key=lambda kv: -kv[1][1]):
        lines.append(f"| `{name}` | {n} | {t:.1f} | {100 * t / total:.1f}% |")
    return "\n".join(lines)


def main():
    p = argparse.ArgumentParser()
    p.add_argument("csv")
    p.add_argument("--after", default=None)
    p.add_argument("--step-launches", type=int, default=0)
    a = p.parse_args()
    launches = read(a.csv)
    ours = [x for x in launches if not x[0].startswith("at::")]
    print(table(launches, "whole run"))
    if a.after and a.step_launches:
        ends = [i for i, x in enumerate(ours) if x[0].startswith(a.after)]
        windows = [i + 1 for i in ends if i + 1 + a.step_launches <= len(ours)
                   and ours[i + a.step_launches][0].startswith(a.after)]
        if windows:
            i = windows[-1]
            print()
            print(table(ours[i:i + a.step_launches], f"one step (library launches {i}..{i + a.step_launches - 1})"))


if __name__ == "__main__":
    main()
