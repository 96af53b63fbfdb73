"""The sampled-run method of the full-size parity tests, checked on the CPU
against the oracle itself: on a BERT-shaped table small enough for the
oracle to run whole (odd tensor offsets, a ragged last chunk), the oracle
run on the sampled runs of whole chunks must give, bit for bit, the
chunk-local state of every sampled element and the parameters and
per-tensor scalars of every tensor a run covers completely, as the oracle
run on the whole table does, over warmup steps, the freeze and compression
steps."""
import numpy as np
import pytest

import fullrun
import oracle
import workload


def _mini(W=4, chunk=512, grad="f32", heavy_every=0):
    t = workload.bert_tensors(3, 96, 384, 700) + [("tail", (37,))]
    return workload.custom("bert_sampled", t, W=W, chunk=chunk, grad=grad, grad_std=1e-3,
                           fan_in_scaled=True, heavy_every=heavy_every)


@pytest.mark.parametrize("kind", ["f32", "bf16", "heavy", "adam+bf16err", "bf16err"])
def test_sampled_runs_reproduce_the_whole_table(kind):
    wl = _mini(grad="bf16" if kind == "bf16" else "f32", heavy_every=5 if kind == "heavy" else 0)
    assert wl.N % 32 != 0 and wl.N % wl.chunk != 0
    tensors, runs = fullrun.plan_for(wl, max_elems=12 * wl.chunk, big=1 << 14)
    assert len(runs) >= 3 and len(tensors) >= 8
    assert runs[-1][1] == wl.K - 1                 # the ragged last chunk is sampled
    opts = dict(variant=int(kind.startswith("adam")), error_storage=int(kind.endswith("bf16err")))
    pl = dict(n_warm=3, n_comp=4, checkpoints=(2, "freeze", 3, 6), **opts)

    # whole table
    full = oracle.Oracle(wl.offsets, wl.numels, wl.W, wl.chunk, wl.hp, workload.gen_params(wl),
                         variant=opts["variant"], err_bf16=opts["error_storage"])
    steps, cps = [], {}
    for step in range(pl["n_warm"] + pl["n_comp"]):
        if step == pl["n_warm"]:
            full.freeze()
            cps["freeze"] = full.snapshot()
        g = workload.grads_for_step(wl, step)
        if step < pl["n_warm"]:
            full.warmup_step(g)
        else:
            full.compress_step(g)
        steps.append(full.snapshot())
        if step in pl["checkpoints"]:
            cps[step] = full.snapshot()

    # sampled runs, two groups as the GPU test splits them
    parts = fullrun.groups(wl, runs, 2)
    rec = {}
    for p in parts:
        rec.update(fullrun.oracle_runs(wl, runs, pl, p))
    C, N = wl.chunk, wl.N
    for r, (k0, k1) in enumerate(runs):
        lo, hi, frags = fullrun.run_table(wl, k0, k1)
        for step, o in enumerate(rec[r]["steps"]):
            f = steps[step]
            for j, (l, a, n, whole) in enumerate(frags):
                if not whole:
                    continue
                for k in ("c_cur", "c_bar") + (("Sx", "Su") if step < pl["n_warm"] else ("R", "r_prev")):
                    assert o[k][j].view(np.uint32) == f[k][l].view(np.uint32), (r, step, k, l)
            if step >= pl["n_warm"]:
                q0, q1 = lo // 32, -(-hi // 32)
                np.testing.assert_array_equal(o["signs_s"], f["signs_s"][q0:q1])
                np.testing.assert_array_equal(o["signs_w"], f["signs_w"][:, q0:q1])
                np.testing.assert_array_equal(o["scale_s"].view(np.uint32),
                                              f["scale_s"][k0:k1 + 1].view(np.uint32))
                np.testing.assert_array_equal(o["scale_w"].view(np.uint32),
                                              f["scale_w"][:, k0:k1 + 1].view(np.uint32))
        for cp, o in rec[r]["checkpoints"].items():
            f = cps[cp]
            for k in ("m", "v", "v_fresh", "e_s"):
                np.testing.assert_array_equal(o[k].view(np.uint32), f[k][lo:hi].view(np.uint32),
                                              err_msg=f"{r} {cp} {k}")
            np.testing.assert_array_equal(o["e_w"].view(np.uint32), f["e_w"][:, lo:hi].view(np.uint32))
            for l, a, n, whole in frags:
                if whole:
                    np.testing.assert_array_equal(o["x"][a:a + n].view(np.uint32),
                                                  f["x"][lo + a:lo + a + n].view(np.uint32))
    del C, N


def test_a_planted_cross_chunk_dependence_is_caught():
    """The comparison has teeth: a run that starts one granule late (so its
    chunks are misaligned with the whole table's) must disagree."""
    wl = _mini()
    tensors, runs = fullrun.plan_for(wl, max_elems=12 * wl.chunk, big=1 << 14)
    k0, k1 = runs[0]
    lo, hi = k0 * wl.chunk + 256, min((k1 + 1) * wl.chunk, wl.N)
    x0 = workload.gen_params(wl, lo, hi)
    o = oracle.Oracle([0], [hi - lo], wl.W, wl.chunk, wl.hp, x0)
    full = oracle.Oracle(wl.offsets, wl.numels, wl.W, wl.chunk, wl.hp, workload.gen_params(wl))
    for step in range(2):
        if step == 1:
            o.freeze()
            full.freeze()
        g = np.stack([workload.gen_grads_range(wl, step, w, lo, hi) for w in range(wl.W)])
        gf = workload.grads_for_step(wl, step)
        if step == 0:
            o.warmup_step(g)
            full.warmup_step(gf)
        else:
            o.compress_step(g)
            full.compress_step(gf)
    assert not np.array_equal(o.e_s.view(np.uint32), full.e_s[lo:hi].view(np.uint32))
