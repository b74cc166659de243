"""Per-item timeline of the cascade kernel on the bench's full three-bank step.

Builds the timeline variant of the library (``build.py --timeline``: the same kernels,
with %globaltimer and clock64 stamps at each hand-off of every work item), runs the
bench workload (qk 22x256x768 + vo 22x768x768 + mlp 22x2816x768, grad pool entry 0,
post-engage scalars) eagerly, and prints a Markdown summary of where each CTA pair's
time goes:

  * the k-loop of every product tile (first k-block landed -> last MMAs issued, plus one
    k-block for the last MMAs to run), and its SM cycles per 64-deep k-block by tile kind;
  * each gap between two product tiles of a pair, split into: the entry reaching the MMA
    issuer (scheduler: dependency wait and hand-off), the accumulator becoming free (the
    epilogue of the tile two back), and the new tile's first k-block landing;
  * the time before a pair's first tile and after its last.

  python -m polynomial_matrix_whitening_gb300.timeline [--reps N]
"""
from __future__ import annotations

import argparse
import os
import statistics
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OPS = {0: "Gram", 1: "first Gram", 2: "bA+cA^2", 3: "X-update", 4: "last X-update"}
BANK_NAMES = ("qk", "vo", "mlp")
(META, TILE, SCHED_TAKE, SCHED_READY, SCHED_PUSH, PROD_FIRST, MMA_TAKEN, MMA_ACC_FREE, MMA_FIRST,
 MMA_LAST, EPI_START, EPI_END, MMA_FIRST_CLK, MMA_LAST_CLK, MMA_WAIT_CLK, PROD_WAIT_CLK) = range(16)


def decode(tl, bank_of_index):
    """Items of one launch as a list of dicts (only the items that were recorded)."""
    items = []
    for t in range(tl.shape[0]):
        r = tl[t]
        if r[SCHED_TAKE] == 0:
            continue
        meta = int(r[META])
        w = (meta >> 16) & 0xffffffff
        tile = int(r[TILE])
        items.append(dict(
            t=t, pair=meta & 0xffff, op=w & 0xff, bank=bank_of_index[(w >> 8) & 0xff], ph=w >> 16,
            mat=meta >> 48, bi=tile & 0xffff, bj=(tile >> 16) & 0xffff, nkb=tile >> 32,
            **{k: int(r[i]) for k, i in (("take", SCHED_TAKE), ("ready", SCHED_READY), ("push", SCHED_PUSH),
                                         ("prod", PROD_FIRST), ("taken", MMA_TAKEN), ("acc", MMA_ACC_FREE),
                                         ("first", MMA_FIRST), ("last", MMA_LAST), ("epi0", EPI_START),
                                         ("epi1", EPI_END), ("c0", MMA_FIRST_CLK), ("c1", MMA_LAST_CLK),
                                         ("mwait", MMA_WAIT_CLK), ("pwait", PROD_WAIT_CLK))}))
    return items


def kind(it):
    return f"{BANK_NAMES[it['bank']]} {OPS[it['op']]} (K={64 * it['nkb']})"


def analyse(items):
    prod = [i for i in items if i["first"] > 0]
    t0 = min(i["take"] for i in items)
    t1 = max(max(i["epi1"], i["last"]) for i in items)
    span = (t1 - t0) / 1e3
    # ns per k-block of each product tile (the last k-block's MMAs run after `last`)
    for i in prod:
        i["kb_ns"] = (i["last"] - i["first"]) / (i["nkb"] - 1) if i["nkb"] > 1 else 0.0
        i["cyc"] = (i["c1"] - i["c0"]) / (i["nkb"] - 1) if i["nkb"] > 1 else 0.0
    med_kb = statistics.median(i["kb_ns"] for i in prod if i["nkb"] > 1)
    pairs = sorted({i["pair"] for i in items})
    acc = dict(kloop=0.0, entry=0.0, accw=0.0, firstkb=0.0, head=0.0, tail=0.0)
    by_next = {}
    by_bank = {}  # pair-time of each bank's product tiles: k-loop + the gap before the tile
    for p in pairs:
        mine = sorted((i for i in prod if i["pair"] == p), key=lambda i: i["first"])
        if not mine:
            acc["head"] += span
            continue
        acc["head"] += (mine[0]["first"] - t0) / 1e3
        end_prev = None
        for i in mine:
            kb = i["kb_ns"] if i["nkb"] > 1 else med_kb
            acc["kloop"] += (i["last"] - i["first"] + kb) / 1e3
            bank = BANK_NAMES[i["bank"]]
            by_bank[bank] = by_bank.get(bank, 0.0) + (i["last"] - i["first"] + kb) / 1e3
            if end_prev is not None:
                by_bank[bank] += max(0, i["first"] - end_prev) / 1e3
                # gap after the previous tile's last MMAs: entry, accumulator, first k-block
                e = max(0, i["taken"] - end_prev) / 1e3
                a = max(0, i["acc"] - max(i["taken"], end_prev)) / 1e3
                f = max(0, i["first"] - max(i["acc"], i["taken"], end_prev)) / 1e3
                acc["entry"] += e
                acc["accw"] += a
                acc["firstkb"] += f
                d = by_next.setdefault(kind(i), [0, 0.0, 0.0, 0.0])
                d[0] += 1
                d[1] += e
                d[2] += a
                d[3] += f
            end_prev = i["last"] + kb
        acc["tail"] += (t1 - end_prev) / 1e3
    n = len(pairs)
    per_pair = {k: v / n for k, v in acc.items()}
    rate = {}
    for i in prod:
        if i["nkb"] > 1:
            rate.setdefault(kind(i), []).append((i["cyc"], i["mwait"] / (i["nkb"] - 1), i["pwait"] / i["nkb"]))
    deps = {}
    for i in items:
        d = deps.setdefault(OPS[i["op"]], [0, 0.0])
        d[0] += 1
        d[1] += (i["ready"] - i["take"]) / 1e3
    return dict(span=span, pairs=n, items=len(items), tiles=len(prod), per_pair=per_pair, rate=rate,
                by_next=by_next, deps=deps, by_bank={k: v / n for k, v in by_bank.items()})


def report(res, cascade_ms, clocks_note):
    pp = res["per_pair"]
    span = res["span"]
    out = []
    out.append(f"Cascade launch: {span:.1f} us from the first item taken to the last tile done "
               f"(CUDA events around the launch: {cascade_ms * 1e3:.1f} us); {res['pairs']} CTA pairs, "
               f"{res['items']} items, {res['tiles']} product tiles. {clocks_note}")
    out.append("")
    out.append("| per CTA pair (mean over pairs) | us | share of the span |")
    out.append("|---|---|---|")
    rows = [("k-loops of product tiles (first k-block landed to last MMAs done)", pp["kloop"]),
            ("gaps: entry not yet with the MMA issuer (dependency wait, hand-off)", pp["entry"]),
            ("gaps: accumulator still in the epilogue", pp["accw"]),
            ("gaps: first k-block of the new tile not yet landed", pp["firstkb"]),
            ("before the pair's first tile", pp["head"]),
            ("after the pair's last tile", pp["tail"])]
    for name, v in rows:
        out.append(f"| {name} | {v:.1f} | {v / span:.1%} |")
    out.append("")
    out.append("| bank | pair-time of its product tiles (k-loop + the gap before each), us per pair | share of the span |")
    out.append("|---|---|---|")
    for k in BANK_NAMES:
        if k in res["by_bank"]:
            out.append(f"| {k} | {res['by_bank'][k]:.1f} | {res['by_bank'][k] / span:.1%} |")
    out.append("")
    out.append("| tile kind | tiles | SM cycles per k-block (median) | of which the MMA issuer waited for operands | producer's wait for a free stage, per k-block | gaps before it: entry / accumulator / first k-block, us (mean) |")
    out.append("|---|---|---|---|---|---|")
    for k in sorted(res["rate"], key=lambda k: -len(res["rate"][k]) * statistics.median(c[0] for c in res["rate"][k])):
        c = res["rate"][k]
        g = res["by_next"].get(k, [0, 0, 0, 0])
        gn = max(g[0], 1)
        out.append(f"| {k} | {len(c)} | {statistics.median(x[0] for x in c):.0f} | "
                   f"{statistics.median(x[1] for x in c):.0f} | {statistics.median(x[2] for x in c):.0f} | "
                   f"{g[1] / gn:.2f} / {g[2] / gn:.2f} / {g[3] / gn:.2f} |")
    out.append("")
    out.append("| phase | items | scheduler's dependency wait, us (sum over items) |")
    out.append("|---|---|---|")
    for k, (cnt, s) in res["deps"].items():
        out.append(f"| {k} | {cnt} | {s:.1f} |")
    return "\n".join(out)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--dump", default=None, help="also save the raw timelines (npz) to this path")
    args = ap.parse_args()
    sys.path.insert(0, ROOT)
    from polynomial_matrix_whitening_gb300 import build as B
    B.build(timeline=True)
    os.environ["ANVIL_LIBRARY"] = "timeline"
    import torch
    from polynomial_matrix_whitening_gb300 import anvil
    from polynomial_matrix_whitening_gb300 import workloads as W
    assert anvil.LIB_PATH.endswith("libanvil_timeline.so"), anvil.LIB_PATH
    dev = torch.device("cuda", 0)
    wl = W.workloads()["full_step"]
    sc = wl.scalars(0)
    banks = [anvil.Bank(torch.from_numpy(wl.grad(j, 0)).to(dev), torch.from_numpy(wl.velocity(j)).to(dev),
                        torch.empty((b.g, b.m, b.n), dtype=torch.bfloat16, device=dev),
                        momentum=sc.momentum, fast_beta=sc.fast_beta, fast_weight=sc.fast_weight,
                        slow_beta=sc.slow_beta) for j, b in enumerate(wl.banks)]
    ws = anvil.alloc_workspace([b.shape for b in banks], device=dev)
    # the cascade walks banks heaviest first: map its bank index back to the call's banks
    runs = anvil.schedule_runs([b.shape for b in banks])
    order = []
    for r in runs:
        if r["bank"] not in order:
            order.append(r["bank"])
    bank_of_index = {q: order[q] for q in range(len(order))}
    for _ in range(3):
        anvil.multi_bank_step(banks, ws)
    torch.cuda.synchronize()
    results, raw = [], []
    for rep in range(args.reps):
        anvil.timeline_clear()
        with anvil.profile(max_records=16) as prof:
            anvil.multi_bank_step(banks, ws)
        torch.cuda.synchronize()
        if anvil.device_error() != anvil.OK:
            raise RuntimeError("device error word set")
        tl = anvil.timeline_read()
        casc = [ms for k, ms in prof.records if k == "cascade"]
        res = analyse(decode(tl, bank_of_index))
        results.append((res, casc[0] if casc else float("nan")))
        raw.append(tl)
    if args.dump:
        np.savez_compressed(args.dump, timelines=np.stack(raw),
                            bank_of_index=np.array([bank_of_index[q] for q in range(len(bank_of_index))]))
    # report the median launch by span
    results.sort(key=lambda r: r[0]["span"])
    res, ms = results[len(results) // 2]
    print(report(res, ms, f"Median of {args.reps} eager steps by span."))


if __name__ == "__main__":
    main()
