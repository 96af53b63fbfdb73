"""Oracle side of the full-size multi-step parity tests (test helper, no
GPU, no torch).

Every quantity of the 1-bit LAMB step except the parameters and the
per-tensor scalars is local to its compression chunk: the warmup moments are
element-wise, and the compression stage's worker momentum, worker and server
errors, sign words, chunk scales and fresh second moment depend only on the
chunk's own elements (1-bit LAMB: background on error-compensated
compression; section 5, where server i owns chunk i).  The parameters of a
tensor depend on its per-tensor coefficient, which the whole tensor
determines (background on LAMB; section 4 summary for the compression-stage
factor).  So the oracle can run a configuration's whole step sequence on a
sample of the flat buffer made of runs of consecutive chunks, each run
covering its chosen tensors completely: every chunk-local value of a run and
every per-tensor value of a tensor that lies inside a run is exactly what the
full-size run computes.  Runs start on chunk boundaries (multiples of the
256-element granule), so the canonical reduction order is unchanged.

The runs are independent problems, so they are spread over processes; this
module holds the per-process work and imports only numpy, the oracle and
the seeded input generator.
"""
from __future__ import annotations

import numpy as np

import oracle
import workload

# Plans: warmup steps, compression steps, and the steps after which the full
# sampled state is compared (a step index counts from 0 over both stages;
# "freeze" is the state right after the variance freeze).
PLANS = {
    "base": dict(n_warm=10, n_comp=10, checkpoints=(9, "freeze", 10, 19)),
    "large": dict(n_warm=10, n_comp=100, checkpoints=(9, "freeze", 10, 19, 109)),
    "large_w32": dict(n_warm=50, n_comp=50, checkpoints=(48, 49, "freeze", 50, 51, 99)),
    "gpt2xl": dict(n_warm=10, n_comp=50, checkpoints=(9, "freeze", 10, 19, 59)),
    # the options on the BERT-Large table, each with its own kernel shape:
    # bfloat16 error storage with each method variant, and 1-bit Adam
    # (variant 1)
    "large:adam+bf16err": dict(n_warm=10, n_comp=20, checkpoints=(9, "freeze", 10, 29),
                               variant=1, error_storage=1),
    "large:bf16err": dict(n_warm=10, n_comp=20, checkpoints=(9, "freeze", 10, 29),
                          error_storage=1),
    "large:adam": dict(n_warm=10, n_comp=20, checkpoints=(9, "freeze", 10, 29), variant=1),
}

# sampled elements per workload (bounds the oracle's CPU time), and the
# largest tensor taken among the table's first and last tensors and the one
# square weight (the W=32 workload's budget goes to its small tensors, where
# the Student-t ones are)
SAMPLE_ELEMS = {"base": 3_000_000, "large": 1_500_000, "large_w32": 1_000_000,
                "gpt2xl": 3_000_000}
BIG = {"base": 4 << 20, "large": 4 << 20, "large_w32": 1 << 16, "gpt2xl": 4 << 20}


def choose_tensors(wl, max_elems: int, big: int):
    """Tensors to cover completely: the first and last few tensors of the
    table (odd-offset tails such as the NSP and decoder biases, the last
    chunk), one square weight, then the small tensors (LayerNorm gains and
    biases, biases) of layers spread evenly, until the chunks holding them
    reach max_elems elements."""
    C, L = wl.chunk, wl.L
    off, num = wl.offsets, wl.numels
    names = [n for n, _ in wl.tensors]

    def chunks_of(l):
        return set(range(int(off[l]) // C, (int(off[l] + num[l]) - 1) // C + 1))

    chosen, ks = [], set()

    def take(l):
        c = chunks_of(l)
        if len(ks | c) * C > max_elems and chosen:
            return False
        chosen.append(l)
        ks.update(c)
        return True

    must = [l for l in range(1, 5) if num[l] <= big]
    must += [l for l in range(L - 9, L) if num[l] <= big]
    sq = [l for l in range(L) if len(wl.tensors[l][1]) == 2
          and wl.tensors[l][1][0] == wl.tensors[l][1][1] and num[l] <= big]
    must += sq[1:2]
    for l in dict.fromkeys(must):
        take(l)
    small = [l for l in range(L) if num[l] <= 2 * C and l not in chosen]
    # spread: every other small tensor first, then the rest
    order = small[::2] + small[1::2]
    for l in order:
        take(l)
    return sorted(chosen), sorted(ks), names


def runs_of(ks, K):
    """Maximal runs of consecutive chunk indices, plus the last chunk."""
    ks = sorted(set(ks) | {K - 1})
    runs = []
    start = prev = ks[0]
    for k in ks[1:]:
        if k != prev + 1:
            runs.append((start, prev))
            start = k
        prev = k
    runs.append((start, prev))
    return runs


def run_table(wl, k0, k1):
    """Local layer table of chunks k0..k1: every tensor's intersection with
    [k0 C, min((k1+1) C, N)), rebased to 0.  Returns (lo, hi, frags) with
    frags = [(global tensor, local offset, numel, whole)]."""
    C, N = wl.chunk, wl.N
    lo, hi = k0 * C, min((k1 + 1) * C, N)
    ends = wl.offsets + wl.numels
    frags = []
    l = int(np.searchsorted(ends, lo, side="right"))
    while l < wl.L and wl.offsets[l] < hi:
        a, b = max(lo, int(wl.offsets[l])), min(hi, int(ends[l]))
        whole = a == wl.offsets[l] and b == ends[l]
        frags.append((l, a - lo, b - a, whole))
        l += 1
    return lo, hi, frags


def plan(name: str):
    """The named workload (a plan name "workload:options" uses the workload
    before the colon), its covered tensors and its runs."""
    base = name.split(":")[0]
    wl = workload.workloads()[base]
    return (wl,) + plan_for(wl, SAMPLE_ELEMS[base], BIG[base])


def plan_for(wl, max_elems: int, big: int):
    tensors, ks, _ = choose_tensors(wl, max_elems, big)
    return tensors, runs_of(ks, wl.K)


def run_cost(wl, lo, hi):
    """Relative host cost of a run: elements, with Student-t elements (one
    generator call each) counted four times."""
    n = hi - lo
    if wl.heavy_every:
        ends = wl.offsets + wl.numels
        for l in np.nonzero(wl.layer_heavy)[0]:
            a, b = max(lo, int(wl.offsets[l])), min(hi, int(ends[l]))
            if b > a:
                n += 3 * (b - a)
    return n


def groups(wl, runs, n_groups: int):
    """Run indices split into n_groups lists of similar cost."""
    cost = [run_cost(wl, *run_table(wl, k0, k1)[:2]) for k0, k1 in runs]
    order = sorted(range(len(runs)), key=lambda i: -cost[i])
    load = [0] * n_groups
    out = [[] for _ in range(n_groups)]
    for i in order:
        g = int(np.argmin(load))
        out[g].append(i)
        load[g] += cost[i]
    return [sorted(g) for g in out if g]


def _snapshot(o):
    return dict(x=o.x.copy(), m=o.m.copy(), v=o.v.copy(), v_fresh=o.v_fresh.copy(),
                e_s=o.e_s.copy(), e_w=o.e_w.copy())


def oracle_runs(wl, runs, pl, run_ids):
    """The whole step sequence of plan pl (warmup steps, compression steps,
    checkpoints) of workload wl on the runs run_ids (indices into runs).
    Returns {run id: record}, record = {"steps": [per-step dict],
    "checkpoints": {step: state}}; per-step dicts hold the sign words and
    chunk scales (compression stage) and the per-tensor scalars of the run's
    fragments."""
    n_warm, n_comp, cps = pl["n_warm"], pl["n_comp"], pl["checkpoints"]
    tables = workload.grad_tables(wl)
    orcs = {}
    for r in run_ids:
        k0, k1 = runs[r]
        lo, hi, frags = run_table(wl, k0, k1)
        x0 = workload.gen_params(wl, lo, hi)
        o = oracle.Oracle([f[1] for f in frags], [f[2] for f in frags], wl.W, wl.chunk, wl.hp, x0,
                          variant=pl.get("variant", 0), err_bf16=pl.get("error_storage", 0))
        orcs[r] = (o, lo, hi, frags)
    out = {r: {"steps": [], "checkpoints": {}} for r in run_ids}
    for step in range(n_warm + n_comp):
        if step == n_warm:
            for r, (o, lo, hi, frags) in orcs.items():
                o.freeze()
                if "freeze" in cps:
                    out[r]["checkpoints"]["freeze"] = _snapshot(o)
        for r, (o, lo, hi, frags) in orcs.items():
            g = np.empty((wl.W, hi - lo), np.float32)
            for w in range(wl.W):
                gw = workload.gen_grads_range(wl, step, w, lo, hi, tables)
                g[w] = workload.bf16_round(gw) if wl.grad == "bf16" else gw
            if step < n_warm:
                o.warmup_step(g)
            else:
                o.compress_step(g)
            rec = dict(c_cur=o.c_cur.copy(), c_bar=o.c_bar.copy())
            if step < n_warm:
                rec.update(Sx=o.Sx.copy(), Su=o.Su.copy())
            else:
                rec.update(R=o.R.copy(), r_prev=o.r_prev.copy(), signs_s=o.signs_s.copy(),
                           scale_s=o.scale_s.copy(), signs_w=o.signs_w.copy(),
                           scale_w=o.scale_w.copy())
            out[r]["steps"].append(rec)
            if step in cps:
                out[r]["checkpoints"][step] = _snapshot(o)
    return out
